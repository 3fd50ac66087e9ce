"""CPU oracle for one speculative-decoding verify round.

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only ``tests/``, ``__graft_entry__.smoke()``
and the ``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import
anything from this package.  The CUDA library never calls it and it never
calls the CUDA library: the two share no code, no tables and no helpers.

What the oracle computes, and where each step comes from (page titles as
printed on the source pages):

* ``quant``  - the affine group-quantized weight: ``w = scale * q + bias`` with
  one fp16 scale and one fp16 bias per group of 64 weights along K.  The
  pages name the "weight group" that the verify kernel dequantizes once
  (mlx-dspark wiki page, "Key techniques"); the packing layout is this
  library's own contract (LSB-first codes in uint32 words).
* ``qmm``    - the skinny verify matmul ``Y = X * W_hat^T`` over the M = 1 + m
  rows of one round (mlx-dspark wiki page, "Architecture": the target runs
  [anchor] + m drafts in one forward), fp64 accumulation, bf16 output; and the
  vocab head with fp32 logits plus per-row max / argmax / sum-exp.
* ``accept`` - the accept step: greedy longest matching prefix (mlx-dspark
  wiki page, "Architecture"; hysenlabs review, "The Problem") and the
  min(1, p/q) rule with residual resampling (mlx-dspark releases page,
  v0.0.2 "Highlights").
* ``philox`` - Philox-4x32-10 (Salmon et al., SC'11) for the uniforms that
  drive sampled acceptance.
* ``glue``   - RMSNorm, residual add and SwiGLU between projections.
* ``chain``  - one verify round of a dense decoder stack built from the above.
* ``cap``    - the draft-cap choice from measured verify costs and a live
  acceptance estimate (PyPI page, "The Apple-Silicon speedup ceiling";
  wiki page, "Key techniques").

Floating point is fp64 unless a step fixes another precision; every place
where the pages are silent and a plain reading was taken is marked
"[reading]".
"""

from . import quant, qmm, accept, philox, glue, chain, cap  # noqa: F401
