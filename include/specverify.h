/*
 * specverify - the verify round of lossless speculative decoding on one GPU.
 *
 * Each round the target model runs the anchor token plus m draft tokens
 * through every linear layer in one pass (mlx-dspark wiki page,
 * "Architecture"), so every projection is a skinny matmul of M = 1 + m rows
 * (1 <= M <= 32; B requests stack their rows into one block) against affine
 * group-quantized weights, and the round ends in an accept step.
 *
 * Conventions for every entry point:
 *   - All array pointers are DEVICE pointers owned by the caller unless the
 *     parameter says "host".  The library allocates no device memory; calls
 *     that need scratch space take a caller-provided workspace whose size comes
 *     from the matching *_workspace_bytes() query, 256-byte aligned.  A
 *     workspace must be zero filled once after allocation (e.g.
 *     cudaMemsetAsync over all of it): it holds a 256 KiB block of counters,
 *     the split-tile partial sums and (for a round) the gate/up partner
 *     values, which every successful call leaves at zero again, so one
 *     workspace (sized for the largest call) can serve any
 *     sequence of calls ordered on one stream.  After a call that reported a
 *     device error, zero it again before reuse.
 *   - bf16 and fp16 values are passed as uint16_t bit patterns.
 *   - Matrices are row-major; ld* is the row stride in elements.
 *   - Every call is asynchronous on `stream` (a cudaStream_t; NULL = the
 *     legacy default stream).  Arguments are validated on the host before
 *     anything is launched: a bad argument returns SV_EINVAL (SV_EUNSUPPORTED
 *     for a valid but unimplemented case) and launches nothing.  A failed
 *     launch returns SV_ECUDA with the CUDA error text in sv_last_error().
 *   - Kernels never trap.  A bounded wait that runs out (about 2 s) records
 *     an error bit in a device word that sv_device_error() reads; results of
 *     that call are then undefined.
 *   - Nothing aborts the process and no C++ exception crosses this boundary.
 *
 * Weight format (mlx-dspark wiki page, "Key techniques": the verify kernel
 * works per weight group; group 64, affine 2-/4-/8-bit codes, fp16 scale and
 * bias per group; PyPI page, "Models": 2-bit targets verify through a
 * multi-row 2-bit matmul):
 *   wq     uint32 [N, K*bits/32]: weight (n, k) is the `bits`-wide field of word
 *          n*(K*bits/32) + k/(32/bits) at bit offset (k % (32/bits))*bits,
 *          least significant field first.
 *   scales fp16 [N, K/64], biases fp16 [N, K/64];  w[n,k] = scale*code + bias.
 *   Requirements: bits in {2, 4, 8}, group == 64, K % 512 == 0, K <= 2^20,
 *   1 <= N <= 2^22, wq, scales and biases 16-byte aligned (the weight rows are streamed by the tensor
 *   memory accelerator in 512-wide k chunks).
 */
#ifndef SPECVERIFY_H
#define SPECVERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  SV_OK = 0,
  SV_EINVAL = 1,        /* bad argument: null/misaligned pointer, bad size */
  SV_EUNSUPPORTED = 2,  /* valid request this build does not implement */
  SV_ECUDA = 3,         /* a CUDA runtime/driver call failed */
  SV_ETIMEOUT = 4       /* a device-side bounded wait ran out (sv_device_error) */
} sv_status;

/* Static text for a status code. */
const char* sv_status_string(int status);
/* Detail of the last non-OK status returned on the calling thread. */
const char* sv_last_error(void);
/* Library version, major*10000 + minor*100 + patch. */
int sv_version(void);
/* Waits for the device, then reads and clears the device error word.
 * Returns SV_OK if no kernel recorded an error, SV_ETIMEOUT otherwise (the
 * raw bits go to *bits when bits != NULL), SV_ECUDA if the device call fails. */
int sv_device_error(unsigned int* bits);
/* Self-test of that path (no counterpart on the pages: a failure-detection
 * check).  Enqueues on `stream` one device-side bounded wait on a barrier
 * that nothing completes, limited to limit_us microseconds (1 .. 1e6); when it
 * runs out the kernel records a timeout bit, exactly as the library's own
 * waits do, and returns: the device faults nothing and stays usable.  The
 * next sv_device_error() then returns SV_ETIMEOUT.  SV_EINVAL for a limit
 * out of range. */
int sv_selftest_bounded_wait(unsigned int limit_us, void* stream);

/* ------------------------------------------------------------------ qmm ---
 * Y[m, n] = sum_k X[m, k] * w[n, k] for one verify projection
 * (PyPI page, "The Apple-Silicon speedup ceiling": verify cost is the
 * quantized matmul over every linear layer; wiki page, "Key techniques":
 * each weight group is dequantized once and reused across all M rows).
 * Arithmetic: fp32 accumulation, output rounded to bf16 (nearest even).
 *   x  bf16 [M, K] with row stride ldx >= K;  y  bf16 [M, N], stride ldy >= N.
 *   residual (optional, may be NULL): bf16 [M, N] with stride ldr; when given,
 *   y = bf16(residual + bf16(x*w^T)), and y may alias residual (in-place add).
 * Workspace: sv_qmm_workspace_bytes(M, N, K, bits) bytes, 256-byte aligned.
 * The result is bitwise reproducible for a given (shape, device). */
size_t sv_qmm_workspace_bytes(int M, int N, int K, int bits);
int sv_qmm_verify(const uint32_t* wq, const uint16_t* scales, const uint16_t* biases, int N, int K, int bits,
                  int group, const uint16_t* x, int ldx, int M, uint16_t* y, int ldy, const uint16_t* residual,
                  int ldr, void* workspace, size_t workspace_bytes, void* stream);

/* Allocation-free sv_qmm_verify (no counterpart on the pages: it serves
 * callers that cannot provide device memory).  Some callers cannot allocate:
 * a plugin inside a host application that owns all device memory, or a
 * runtime that forbids cudaMalloc after start-up because it can synchronize
 * the device.  This form takes no workspace; its scratch lives in one
 * device array built into the library, sv_qmm_noalloc_scratch_bytes()
 * bytes (4 MiB) on every GPU that loads the library, held until the process
 * exits.  Calls whose scratch would exceed it (roughly M = 32 with K above
 * 20k) return SV_EUNSUPPORTED with the needed size in sv_last_error().
 * Same arguments and results as sv_qmm_verify, minus the workspace.
 *   - The array and this library's kernels get their device memory when
 *     CUDA loads the library's module on a device, which with CUDA's default
 *     lazy loading happens at the first call there: make one call per
 *     device at start-up, outside any no-allocation window and before any
 *     stream capture.  Every call looks the array's device address up again
 *     (cheap once loaded), so a context rebuilt after cudaDeviceReset is
 *     handled.
 *   - Every call shares the array and clears its own counters first; calls
 *     that overlap on the GPU (other streams, or other host threads) race on
 *     the array, so order them on one stream.
 *   - Allocates nothing: no cudaMalloc, no cudaFree, no allocating library call. */
size_t sv_qmm_noalloc_scratch_bytes(void);
int sv_qmm_verify_noalloc(const uint32_t* wq, const uint16_t* scales, const uint16_t* biases, int N, int K, int bits,
                          int group, const uint16_t* x, int ldx, int M, uint16_t* y, int ldy,
                          const uint16_t* residual, int ldr, void* stream);

/* Split form of sv_qmm_verify for chains of projections.  sv_qmm_prepare
 * converts one activation block into the layout the matmul kernel streams
 * (kept in the workspace); each later sv_qmm_run / sv_lm_head_run with the
 * same M, K and bits consumes it, so several projections of one input
 * share one preparation.  The preparation can fuse the step that produces
 * the activations:
 *   SV_PREP_PLAIN    x as given (bf16 [M, K], stride ldx)
 *   SV_PREP_RMSNORM  x / sqrt(mean(x^2) + eps) * weight, weight bf16 [K] or NULL = 1;
 *                    the row scale is applied in fp32 to the matmul output, so
 *                    the normalized row is never rounded to bf16 (the result
 *                    differs from sv_rmsnorm + SV_PREP_PLAIN only by that rounding)
 *   SV_PREP_SWIGLU   bf16(silu(x) * x2) with x2 bf16 [M, K] (stride ldx2); bit-identical
 *                    to sv_swiglu followed by SV_PREP_PLAIN
 * Workspace: sv_qmm_workspace_bytes() of the run that follows. */
enum { SV_PREP_PLAIN = 0, SV_PREP_RMSNORM = 1, SV_PREP_SWIGLU = 2 };
int sv_qmm_prepare(const uint16_t* x, int ldx, int M, int K, int bits, int mode, const uint16_t* x2, int ldx2,
                   const uint16_t* rms_weight, float eps, void* workspace, size_t workspace_bytes, void* stream);
int sv_qmm_run(const uint32_t* wq, const uint16_t* scales, const uint16_t* biases, int N, int K, int bits, int group,
               int M, uint16_t* y, int ldy, const uint16_t* residual, int ldr, void* workspace,
               size_t workspace_bytes, void* stream);

/* Gather form for mixture-of-experts targets (PyPI page, "Results at a
 * glance": on an MoE target every verify row pulls in its own set of
 * experts; wiki page, "Key techniques": each weight group is dequantized once
 * and reused across rows).  P (row, expert) pairs:
 *   Y[p, :] = X[pair_rows[p], :] * W_{pair_experts[p]}^T,   p = 0 .. P-1,
 * with the arithmetic of sv_qmm_verify.  The experts are stacked along N:
 * wq [E*N, K*bits/32], scales / biases [E*N, K/64] (expert e owns rows
 * e*N .. e*N + N - 1), in the weight format above.  x bf16 [M, K] (stride
 * ldx), M <= 32; pair_rows and pair_experts are DEVICE int32 [P] (1 <= P <=
 * 1024); y bf16 [P, N] (stride ldy).  The pairs are grouped by expert on the
 * device: every selected expert is streamed once and applied to all rows
 * routed to it.  An expert may receive at most M pairs; a pair with a row
 * outside [0, M) or an expert outside [0, E), or an expert's pairs beyond M,
 * leave their output rows untouched and set the bad-input bit that
 * sv_device_error() reports.  1 <= E <= 4096.
 * Workspace: sv_gather_qmm_workspace_bytes(P, M, N, K, E, bits), 256-byte
 * aligned; no zero-fill needed. */
size_t sv_gather_qmm_workspace_bytes(int P, int M, int N, int K, int E, int bits);
int sv_gather_qmm(const uint32_t* wq, const uint16_t* scales, const uint16_t* biases, int E, int N, int K, int bits,
                  int group, const uint16_t* x, int ldx, int M, const int32_t* pair_rows, const int32_t* pair_experts,
                  int P, uint16_t* y, int ldy, void* workspace, size_t workspace_bytes, void* stream);

/* -------------------------------------------------------------- lm_head ---
 * The vocab head of the round with its row softmax statistics fused in
 * (wiki page, "Architecture": the draft is compared against the target's own
 * logits; "Design decisions": verification keeps the full head transform).
 *   logits  fp32 [M, V], stride ldl >= V (no 16-bit rounding).
 *   row_max fp32 [M], row_argmax int32 [M] (lowest index attaining the max),
 *   row_sumexp fp32 [M] = sum_v exp((logits - row_max) / T), written only when
 *   temperature > 0 (may be NULL when temperature == 0).  Any of the three
 *   row outputs may be NULL to skip it.
 * temperature >= 0; 0 means greedy.
 * Workspace: sv_lm_head_workspace_bytes(M, V, K, bits). */
size_t sv_lm_head_workspace_bytes(int M, int V, int K, int bits);
int sv_lm_head_verify(const uint32_t* wq, const uint16_t* scales, const uint16_t* biases, int V, int K, int bits,
                      int group, const uint16_t* x, int ldx, int M, float temperature, float* logits, int ldl,
                      float* row_max, float* row_sumexp, int32_t* row_argmax, void* workspace,
                      size_t workspace_bytes, void* stream);
/* The vocab head on activations prepared by sv_qmm_prepare (same M, K, bits). */
int sv_lm_head_run(const uint32_t* wq, const uint16_t* scales, const uint16_t* biases, int V, int K, int bits,
                   int group, int M, float temperature, float* logits, int ldl, float* row_max, float* row_sumexp,
                   int32_t* row_argmax, void* workspace, size_t workspace_bytes, void* stream);

/* --------------------------------------------------------------- accept ---
 * Accept step of one round (B = 1) or of B independent requests.
 * Greedy (temperature == 0; wiki page, "Architecture"; hysenlabs review,
 * "The Problem"): a = first i < m with draft[i] != argmax(logits[i]) (a = m if
 * none); out_tokens = draft[0..a-1] followed by argmax(logits[a]); out_len = a+1.
 * Sampled (temperature > 0; releases page, v0.0.2 "Highlights"): with
 * p_i = softmax(logits[i] / T), draft i is accepted iff u[i] < p_i[d]/q_i[d]
 * (q_i[d] == 0 accepts).  At the first rejection i the committed token is the
 * smallest k whose cumulative residual max(0, p_i - q_i) (index order) exceeds
 * u[m] times its total (a zero residual falls back to p_i); if all m drafts
 * are accepted the bonus token is drawn the same way from p_m.
 *   logits fp32 [m+1, V] (stride ldl); q fp32 [m, V] draft probabilities
 *   (stride ldq; unused and may be NULL when T == 0); draft int32 [m] token ids
 *   in [0, V); u fp32 [m+1] uniforms in [0, 1) (may be NULL when T == 0).
 *   row_max, row_sumexp, row_argmax: the lm_head row outputs for these rows.
 *   They may all be NULL, in which case the call computes them itself (one
 *   more pass over the logits); they must all be given or all be NULL.
 *   out_len int32 [1]; out_tokens int32 [m+1] (entries past out_len untouched).
 * 0 <= m <= 31, 2 <= V <= 2^24.
 * Workspace: sv_accept_workspace_bytes(B, max_rows), max_rows = total logits rows. */
size_t sv_accept_workspace_bytes(int B, int max_rows);
int sv_spec_accept(const float* logits, int ldl, const float* row_max, const float* row_sumexp,
                   const int32_t* row_argmax, const float* q, int ldq, const int32_t* draft, int m, int V,
                   float temperature, const float* u, int32_t* out_len, int32_t* out_tokens, void* workspace,
                   size_t workspace_bytes, void* stream);
/* Batched form (PyPI page, "Concurrent throughput": B requests share one
 * forward, each accepts and rolls back on its own).  row_offsets is a HOST
 * array int32 [B+1]: request b owns logits rows [row_offsets[b], row_offsets[b+1])
 * (m_b + 1 rows, 0 <= m_b <= 31), the q and draft rows starting at
 * row_offsets[b] - b (m_b of them), uniforms u[row_offsets[b] .. +m_b], and
 * writes out_len[b] and out_tokens[row_offsets[b] .. +m_b].  1 <= B <= 256. */
int sv_spec_accept_batched(int B, const int32_t* row_offsets, const float* logits, int ldl, const float* row_max,
                           const float* row_sumexp, const int32_t* row_argmax, const float* q, int ldq,
                           const int32_t* draft, int V, float temperature, const float* u, int32_t* out_len,
                           int32_t* out_tokens, void* workspace, size_t workspace_bytes, void* stream);

/* Accept with a truncated target (releases page, v0.1.0 "Highlights":
 * lossless top-p / top-k, the truncation applied to both the draft and the
 * target so the output is an exact sample of the truncated target).  As
 * sv_spec_accept_batched, except that for T > 0 every logits row's target
 * p = softmax(z / T) is first truncated: tokens are ordered by logit, largest
 * first, ties to the lower index; top_k > 0 keeps the first top_k (0 = no
 * limit), then top_p keeps the shortest prefix of those whose share of their
 * mass reaches top_p (1 = no limit); the kept mass is renormalised and every
 * other token has probability 0.  A draft token outside the kept set is
 * rejected.  q must be the distribution the drafts were actually drawn from
 * (truncate it with sv_truncate_probs to apply the same rule on the draft
 * side).  Greedy rounds (T == 0) are unaffected: the argmax is always kept.
 * top_k >= 0, 0 < top_p <= 1.  Workspace: sv_accept_workspace_bytes(). */
int sv_spec_accept_truncated(int B, const int32_t* row_offsets, const float* logits, int ldl, const float* row_max,
                             const float* row_sumexp, const int32_t* row_argmax, const float* q, int ldq,
                             const int32_t* draft, int V, float temperature, const float* u, int top_k, float top_p,
                             int32_t* out_len, int32_t* out_tokens, void* workspace, size_t workspace_bytes,
                             void* stream);
/* The same truncation rule on probability rows (the draft side): each row of
 * probs fp32 [rows, V] (stride ldp) is ordered by value (ties to the lower
 * index), truncated by top_k / top_p and renormalised into out (stride ldo;
 * out may equal probs, otherwise it must not overlap it).  No workspace. */
int sv_truncate_probs(const float* probs, int ldp, float* out, int ldo, int rows, int V, int top_k, float top_p,
                      void* stream);
/* Log-probabilities of the target (releases page, v0.2.0 "Highlights":
 * logprobs / top_logprobs, the chosen and the top target log-probabilities
 * per token).  Per row of logits fp32 [rows, V] (stride ldl), at temperature T
 * (T == 0: T = 1): log p_v = (z_v - max) / T - log sum_k exp((z_k - max) / T),
 * in fp64, stored fp32.  chosen int32 [rows] (may be NULL) -> chosen_logprob
 * fp32 [rows] (NaN for an index outside [0, V)); top_n in [0, 32] -> top_ids
 * int32 [rows, top_n] and top_logprobs fp32 [rows, top_n], ordered by logit
 * (largest first, ties to the lower index).  No workspace. */
int sv_logprobs(const float* logits, int ldl, int rows, int V, float temperature, const int32_t* chosen, int top_n,
                float* chosen_logprob, int32_t* top_ids, float* top_logprobs, void* stream);

/* --------------------------------------------------------------- philox ---
 * n uniforms in [0, 1) from Philox-4x32-10 (Salmon et al., SC'11): element i is
 * word (offset+i) % 4 of Philox(counter = (b lo, b hi, subsequence lo,
 * subsequence hi), key = (seed lo, seed hi)), b = (offset+i) / 4, mapped to
 * (word >> 8) * 2^-24.  Independent requests use distinct subsequences.
 *   out fp32 [n], n >= 0. */
int sv_philox_uniforms(uint64_t seed, uint64_t subsequence, uint64_t offset, int n, float* out, void* stream);

/* ----------------------------------------------------------------- glue ---
 * Row-wise steps between projections of a dense block (the pages give no
 * layer internals; these are the usual RMSNorm / residual / SwiGLU).  fp32
 * arithmetic, bf16 storage, one rounding per output.
 *   sv_rmsnorm:   y = x / sqrt(mean(x^2) + eps) * weight   (weight bf16 [H] or NULL = 1)
 *   sv_residual_add: h = h + t
 *   sv_swiglu:    s = silu(g) * u,  silu(g) = g / (1 + exp(-g))
 * M <= 4096 rows, H (or I) >= 1. */
int sv_rmsnorm(const uint16_t* x, int ldx, int M, int H, const uint16_t* weight, float eps, uint16_t* y, int ldy,
               void* stream);
int sv_residual_add(uint16_t* h, int ldh, const uint16_t* t, int ldt, int M, int H, void* stream);
int sv_swiglu(const uint16_t* g, int ldg, const uint16_t* u, int ldu, int M, int I, uint16_t* s, int lds,
              void* stream);

/* --------------------------------------------------------- verify round ---
 * One whole verify round of a dense target whose every linear layer is
 * group-quantized (wiki page, "Architecture": the target runs [anchor] + m
 * drafts in one forward, then the accept step; PyPI page, "The Apple-Silicon
 * speedup ceiling": verify cost is the quantized matmul over every layer).
 * The pages give no layer internals; the body used here is
 *   h += o(q(RMSNorm(h)))                       (q feeds o: no attention state)
 *   h += down(silu(gate(a)) * up(a)),  a = RMSNorm(h)
 * with RMSNorm weight 1.0 and k, v computed alongside q and unused, followed
 * by a = RMSNorm(h), the vocab head (sv_lm_head_run) and the accept step
 * (sv_spec_accept_batched semantics).  All weights use model->bits, group 64.
 *
 * sv_qweight: one quantized matrix [N, K] in the format above (device pointers).
 * sv_layer:   qkv  = q | k | v stacked along N (first q_dim rows are q), K = hidden
 *             o    = [hidden, q_dim]
 *             gate_up = [2*inter, hidden], gate and up rows interleaved in blocks
 *                    of 64: rows 128j .. 128j+63 are gate rows 64j .. 64j+63 and
 *                    rows 128j+64 .. 128j+127 the matching up rows
 *             down = [hidden, inter]
 *             hidden, q_dim and inter must be multiples of 512.
 * sv_model:   `layers` is a HOST array of n_layers entries; every layer's qkv
 *             has the same N; lm_head = [vocab, hidden].
 *
 * sv_verify_round enqueues the whole round on `stream` as four launches
 * (input preparation, all 4 * n_layers + 1 projections in one persistent
 * cooperative kernel, the row-statistics merge, the accept step); it can be
 * captured into a CUDA graph.  At most 67 layers.  Arguments:
 *   plan    the model's round plan (device, from sv_round_plan_init below).
 *   B, row_offsets (HOST int32 [B+1]): requests stacked into M = row_offsets[B]
 *     rows, 1 <= M <= 32, each as in sv_spec_accept_batched.
 *   hidden  bf16 [M, hidden] (stride ldh): the rows' input hidden states;
 *     updated in place to the final residual stream.
 *   temperature, q (fp32, stride ldq), draft (int32), u (fp32): as in
 *     sv_spec_accept_batched.
 *   logits  fp32 [M, vocab] (stride ldl): the round's target logits.
 *   out_len int32 [B], out_tokens int32 [M]: the accept result.  These two
 *     may also be pinned host memory that the device can address (as from
 *     cudaHostAlloc on a system with unified addressing): the accept step
 *     then writes the result straight to the host, with no copy to order
 *     after the round.
 *   event_start, event_stop: optional cudaEvent_t (NULL to skip) recorded on
 *     `stream` just before and after the launch that runs all the projections,
 *     for timing it (recording them adds a dependency that delays that launch
 *     by the previous launch's drain).
 *   accept_wait_event: optional cudaEvent_t (NULL to skip): `stream` waits
 *     for it just before the accept step, the only launch that reads q, draft
 *     and u, so a caller can copy those in on another stream while the
 *     projections run (no counterpart on the pages: a pipelining hook).  In a
 *     stream capture the event must be recorded in the same capture.
 * Workspace: sv_round_workspace_bytes(model, M) bytes (zero-fill rule above). */
typedef struct {
  const uint32_t* wq;
  const uint16_t* scales;
  const uint16_t* biases;
  int N, K;
  const void* packed;  /* optional unit-packed copy from sv_qmm_pack (device, 16-byte aligned), or NULL */
} sv_qweight;
typedef struct {
  sv_qweight qkv, o, gate_up, down;
} sv_layer;
typedef struct {
  int n_layers, hidden, q_dim, inter, vocab, bits;
  float rms_eps;
  const sv_layer* layers;
  sv_qweight lm_head;
} sv_model;

size_t sv_round_workspace_bytes(const sv_model* model, int rows);

/* Unit-packed weights (optional, for sv_verify_round).  The verify matmul
 * streams a weight in units of 64 rows x 512 k; sv_qmm_pack writes a copy of
 * one quantized weight [N, K] in which every unit is one contiguous block
 * (the unit's codes in the shared-memory order the kernel reads, then its
 * scales, then its biases; units tile-major, k-minor; rows beyond N padded
 * with zeros), so the kernel fetches a unit with one bulk copy.  This is a
 * relayout of the same bytes, done once outside the timed path; results are
 * bitwise the same as from the canonical weight.  Set sv_qweight.packed to
 * use it.  sv_qmm_pack_bytes returns ceil(N/64)*64 * K * (bits/8 + 4/64)
 * bytes, or 0 for unsupported sizes (K a multiple of 512).  sv_qmm_pack
 * validates like sv_qmm_verify, launches one kernel on `stream`, and writes
 * only `packed` (caller-owned device memory, 16-byte aligned).  The pages
 * have no counterpart: their weights are used in the canonical layout, and
 * this copy only changes where the same bytes sit. */
size_t sv_qmm_pack_bytes(int N, int K, int bits);
int sv_qmm_pack(const uint32_t* wq, const uint16_t* scales, const uint16_t* biases, int N, int K, int bits, int group,
                void* packed, size_t packed_bytes, void* stream);

/* Round plan: the TMA descriptors of every projection of `model`, built once
 * per model in caller-owned device memory of sv_round_plan_bytes(model) bytes
 * (256-byte aligned).  sv_round_plan_init checks the model (as
 * sv_verify_round does), encodes the descriptors and copies them to `plan`
 * synchronously, so it must not be called while a stream is being captured.
 * The library remembers the weight pointers and shapes each plan was built
 * for; sv_verify_round refuses (SV_EINVAL) a plan built for another model.
 * Rebuild the plan whenever a weight pointer changes.  sv_round_plan_bytes
 * returns 0 for a null model or more than 67 layers. */
size_t sv_round_plan_bytes(const sv_model* model);
int sv_round_plan_init(const sv_model* model, void* plan, size_t plan_bytes);

int sv_verify_round(const sv_model* model, const void* plan, int B, const int32_t* row_offsets, uint16_t* hidden, int ldh,
                    float temperature, const float* q, int ldq, const int32_t* draft, const float* u, float* logits,
                    int ldl, int32_t* out_len, int32_t* out_tokens, void* workspace, size_t workspace_bytes,
                    void* stream, void* event_start, void* event_stop, void* accept_wait_event);

/* ------------------------------------------------------- draft-cap control ---
 * Host-only (no device work, callable without a GPU).  PyPI page, "The
 * Apple-Silicon speedup ceiling": throughput is about A / (drafter + overhead
 * + verify cost) for accept length A and draft cap C, with the verify cost of
 * a wider round measured rather than assumed; wiki page, "Key techniques"
 * (hardware-aware auto-calibration): a controller picks each round's cap from
 * the measured curves and a live acceptance estimate, with expected committed
 * tokens 1 + sum_{i=1}^{C} p^i, and parks speculation (cap 0) when it loses;
 * PyPI page, "Tuning" (--max-draft auto): while parked, plain steps plus
 * periodic probe rounds keep the estimate current.
 *   verify_us[C]  measured device time of a verify round of width M = 1 + C
 *                 (e.g. sv_verify_round timed at every M), C = 0..max_cap, > 0;
 *   draft_us[C]   the drafter's cost of a block of C drafts (draft_us[0] is
 *                 normally 0), >= 0;  overhead_us  per-round host overhead.
 * A round's cost is draft_us[C] + overhead_us + verify_us[C]; the best cap
 * maximises E(C) / cost(C), E(C) = sum_{i=0}^{C} p^i, smallest C on ties.
 * The acceptance estimate p = S / (S + F), where a round that verified C
 * drafts and accepted a adds a to S and [a < C] to F through an EWMA of
 * weight alpha (the maximum-likelihood estimate of a geometric acceptance
 * model); the prior p0 counts as one round.  The struct is caller-owned; its
 * state fields are written by the calls below.  Errors: SV_EINVAL. */
#define SV_CAP_MAX 31
typedef struct {
  int max_cap;                        /* 0..SV_CAP_MAX */
  double verify_us[SV_CAP_MAX + 1];
  double draft_us[SV_CAP_MAX + 1];
  double overhead_us;
  double alpha;                       /* EWMA weight of the newest round, (0, 1] */
  int probe_every;                    /* while parked: one probe round every probe_every rounds */
  int probe_cap;                      /* cap of a probe round, 1..max_cap */
  double S, F;                        /* state: EWMA successes and failures */
  int parked, since_probe;            /* state */
} sv_cap_controller;
/* 1 + p + ... + p^cap (NAN for p outside [0, 1] or cap < 0). */
double sv_expected_committed(double p, int cap);
/* The best cap for a given p and its rate (committed tokens per microsecond). */
int sv_best_cap(double p, int max_cap, const double* verify_us, const double* draft_us, double overhead_us, int* cap,
                double* rate);
/* End of the cheap verify region (PyPI page, "Results at a glance"): the widest
 * M such that verify_us[c] <= (1 + tol) * verify_us[0] for every c < M. */
int sv_verify_knee(const double* verify_us, int n, double tol, int* width);
int sv_cap_init(sv_cap_controller* ctl, int max_cap, const double* verify_us, const double* draft_us,
                double overhead_us, double alpha, int probe_every, int probe_cap, double p0);
/* Cap for the next round (0 = a plain step). */
int sv_cap_next(sv_cap_controller* ctl, int* cap);
/* Record a round that verified `cap` drafts and accepted `accepted` of them. */
int sv_cap_update(sv_cap_controller* ctl, int cap, int accepted);
/* The current acceptance estimate S / (S + F). */
double sv_cap_acceptance(const sv_cap_controller* ctl);

#ifdef __cplusplus
}
#endif

#endif /* SPECVERIFY_H */
