"""The fused preparation modes and the whole verify round against the oracle."""

import numpy as np
import pytest
import torch

from oracle import accept as oa, chain, glue, qmm as oq, quant
import synthetic
from synthetic import model as _model
from tests._util import assert_close_bf16, assert_close_rms, dev_bf16, host_bf16_bits, host_f32_of_bf16, sub_weight

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("M", [1, 8, 17])
def test_fused_prepare_matches_unfused(lib, bits, M):
    r = synthetic.rng(1200 + M + bits)
    K, N = 4096, 1024
    w = _model.to_device(synthetic.quant_weight(r, N, K, bits, synthetic.LARGE_8BIT))
    h = dev_bf16(synthetic.activations(r, M, K, 5.0))
    u = dev_bf16(synthetic.activations(r, M, K, 2.0))
    ws = lib.workspace(lib.qmm_workspace_bytes(M, N, K, bits))
    # RMSNorm fused (row scale applied to the output) vs standalone RMSNorm then matmul
    lib.qmm_prepare(h, K, bits, mode=1, eps=1e-6, workspace=ws)
    y_fused = lib.qmm_run(w["wq"], w["scales"], w["biases"], K, bits, M, workspace=ws)
    y_ref = lib.qmm_verify(w["wq"], w["scales"], w["biases"], K, bits, lib.rmsnorm(h))
    torch.cuda.synchronize()
    assert_close_bf16(host_f32_of_bf16(y_fused), host_f32_of_bf16(y_ref), what="rmsnorm fused")
    # ... against the oracle's RMSNorm -> matmul, and its folded form (one rounding of the output)
    hw = _model.host_copy(w)
    want = oq.qmm_verify(hw["wq"], hw["scales"], hw["biases"], K, bits, glue.rmsnorm(host_bf16_bits(h)))
    assert_close_bf16(host_f32_of_bf16(y_fused), quant.bf16_bits_to_f32(want), what="rmsnorm fused vs oracle")
    hw["K"], hw["bits"] = K, bits
    folded = quant.bf16_bits_to_f32(chain.project_normed(hw, host_bf16_bits(h)))
    assert_close_bf16(host_f32_of_bf16(y_fused), folded, what="rmsnorm fused vs folded oracle")
    # SwiGLU fused vs standalone
    lib.qmm_prepare(h, K, bits, mode=2, x2=u, workspace=ws)
    y_fused = lib.qmm_run(w["wq"], w["scales"], w["biases"], K, bits, M, workspace=ws)
    y_ref = lib.qmm_verify(w["wq"], w["scales"], w["biases"], K, bits, lib.swiglu(h, u))
    torch.cuda.synchronize()
    assert torch.equal(y_fused, y_ref)
    assert lib.device_error() == 0


def _round(lib, model, rows_offsets, h0, T, q=None, draft=None, u=None):
    M = int(rows_offsets[-1])
    V = model.vocab
    hidden = h0.clone()
    logits = torch.empty((M, V), dtype=torch.float32, device="cuda")
    out_len = torch.zeros(len(rows_offsets) - 1, dtype=torch.int32, device="cuda")
    out_tokens = torch.full((M,), -1, dtype=torch.int32, device="cuda")
    ws = lib.workspace(lib.round_workspace_bytes(model, M))
    lib.verify_round(model, rows_offsets, hidden, T, logits, out_len, out_tokens, ws, q=q, draft=draft, u=u)
    torch.cuda.synchronize()
    return hidden, logits, out_len.cpu().numpy(), out_tokens.cpu().numpy()


TINY = dict(hidden=1024, q_dim=1024, kv_dim=512, inter=2048, vocab=1000)


@pytest.mark.parametrize("bits", [4, 2])
@pytest.mark.parametrize("T", [0.0, 1.0])
def test_tiny_model_round_matches_oracle_chain(lib, T, bits):
    n_layers, m = 3, 7
    stats = synthetic.TINY_2BIT if bits == 2 else synthetic.TINY_4BIT
    layers, head = _model.host_model(1300 + bits, n_layers, bits=bits, stats=stats, **TINY)
    dl = _model.device_layers(layers)
    dh = _model.to_device(head)
    r = synthetic.rng(1301)
    h0 = synthetic.activations(r, m + 1, TINY["hidden"])
    hs, logits_or, _, am_or, _ = chain.round_logits(h0, layers, head, T)
    offs = [0, m + 1]
    for depth in range(1, n_layers + 1):      # per-layer hidden state via prefix models
        model = lib.make_model(dl[:depth], dh, TINY["hidden"], TINY["q_dim"], TINY["inter"], TINY["vocab"], bits)
        draft = synthetic.agreeing_drafts(r, am_or[:m], TINY["vocab"])
        z_q = None
        q = u = None
        if T > 0:
            _, z_q = synthetic.logits_and_draft_probs(r, m, TINY["vocab"])
            q = torch.from_numpy(z_q).cuda()
            u = torch.from_numpy(synthetic.accept_uniforms(r, m + 1)).cuda()
        hidden, logits, n, toks = _round(lib, model, offs, dev_bf16(h0), T, q=q,
                                         draft=torch.from_numpy(draft).cuda(), u=u)
        assert_close_bf16(host_f32_of_bf16(hidden), quant.bf16_bits_to_f32(hs[depth - 1]),
                         what="hidden after %d layers" % depth)
    lg = logits.cpu().numpy()
    assert_close_rms(lg, logits_or, what="logits")
    # accept parity on identical (GPU) logits
    if T > 0:
        det = oa.sampled_accept_detail(lg, z_q, draft, T, u.cpu().numpy())
        want = (det["out_len"], det["tokens"])
    else:
        want = oa.greedy_accept(lg, draft)
    assert (int(n[0]), toks[:n[0]].tolist()) == tuple(want)
    assert lib.device_error() == 0


def test_batched_round_four_requests(lib):
    """Continuous-batching shape: 4 requests x (1 + 7) rows in one round, T = 1."""
    layers, head = _model.host_model(1400, 2, bits=8, stats=synthetic.LARGE_8BIT, **TINY)
    model = lib.make_model(_model.device_layers(layers), _model.to_device(head), TINY["hidden"], TINY["q_dim"],
                           TINY["inter"], TINY["vocab"], 8)
    r = synthetic.rng(1401)
    B, m = 4, 7
    offs = [b * (m + 1) for b in range(B + 1)]
    h0 = synthetic.activations(r, B * (m + 1), TINY["hidden"])
    qs = [synthetic.logits_and_draft_probs(r, m, TINY["vocab"])[1] for _ in range(B)]
    drafts = [synthetic.sample_drafts(r, q) for q in qs]
    us = [lib.philox_uniforms(99, b, 0, m + 1) for b in range(B)]
    hidden, logits, n, toks = _round(lib, model, offs, dev_bf16(h0), 1.0,
                                     q=torch.from_numpy(np.concatenate(qs)).cuda(),
                                     draft=torch.from_numpy(np.concatenate(drafts)).cuda(), u=torch.cat(us))
    lg = logits.cpu().numpy()
    _, logits_or, _, _, _ = chain.round_logits(h0, layers, head, 1.0)
    assert_close_rms(lg, logits_or, what="batched logits")
    want = oa.spec_accept_batched(lg, np.concatenate(qs), drafts, offs, 1.0, [x.cpu().numpy() for x in us])
    for b in range(B):
        assert (int(n[b]), toks[offs[b]:offs[b] + n[b]].tolist()) == tuple(want[b])


def test_round_accept_inputs_on_a_side_stream(lib):
    """q, draft and u copied in from pinned host memory on another stream while the
    projections run, the accept step waiting for them (accept_wait_event), inside a
    captured CUDA graph: the same bits as the round with its inputs resident."""
    layers, head = _model.host_model(1500, 2, bits=8, stats=synthetic.LARGE_8BIT, **TINY)
    model = lib.make_model(_model.device_layers(layers), _model.to_device(head), TINY["hidden"], TINY["q_dim"],
                           TINY["inter"], TINY["vocab"], 8)
    r = synthetic.rng(1501)
    m = 7
    M = m + 1
    h0 = synthetic.activations(r, M, TINY["hidden"])
    qn = synthetic.logits_and_draft_probs(r, m, TINY["vocab"])[1]
    dn = synthetic.sample_drafts(r, qn)
    un = synthetic.accept_uniforms(r, M)
    # reference: everything resident before the call
    ref = _round(lib, model, [0, M], dev_bf16(h0), 1.0, q=torch.from_numpy(qn).cuda(),
                 draft=torch.from_numpy(dn).cuda(), u=torch.from_numpy(un).cuda())
    # the pipelined form, captured once and replayed
    hq, hd, hu = (torch.from_numpy(a).pin_memory() for a in (qn, dn, un))
    q, d, u = (torch.empty_like(a, device="cuda") for a in (hq, hd, hu))
    hidden = dev_bf16(h0)
    h_init = hidden.clone()
    logits = torch.zeros((M, TINY["vocab"]), dtype=torch.float32, device="cuda")
    out_len = torch.zeros(1, dtype=torch.int32, device="cuda")
    out_tokens = torch.full((M,), -1, dtype=torch.int32, device="cuda")
    ws = lib.workspace(lib.round_workspace_bytes(model, M))
    ready = torch.cuda.Event()
    main, side = torch.cuda.Stream(), torch.cuda.Stream()

    def step():
        side.wait_stream(main)
        with torch.cuda.stream(side):
            for dev, host in ((q, hq), (d, hd), (u, hu)):
                dev.copy_(host, non_blocking=True)
            ready.record(side)
        with torch.cuda.stream(main):
            hidden.copy_(h_init)
            lib.verify_round(model, [0, M], hidden, 1.0, logits, out_len, out_tokens, ws, q=q, draft=d, u=u,
                             stream=main, accept_wait=ready)

    main.wait_stream(torch.cuda.current_stream())
    step()                                   # eager once (kernel attributes are set outside capture)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=main):
        step()
    for _ in range(2):
        q.zero_()
        d.zero_()
        u.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(hidden, ref[0]) and torch.equal(logits, ref[1])
        assert (out_len.cpu().numpy() == ref[2]).all() and (out_tokens.cpu().numpy() == ref[3]).all()
    assert lib.device_error() == 0



def test_round_writes_its_result_to_pinned_host_memory(lib):
    """out_len / out_tokens in pinned host memory the device can address: the
    accept step writes the result to the host directly, eagerly and from a
    captured graph, with the same values as device outputs."""
    layers, head = _model.host_model(1510, 2, bits=8, stats=synthetic.LARGE_8BIT, **TINY)
    model = lib.make_model(_model.device_layers(layers), _model.to_device(head), TINY["hidden"], TINY["q_dim"],
                           TINY["inter"], TINY["vocab"], 8)
    r = synthetic.rng(1511)
    m, B = 5, 2
    M = B * (m + 1)
    offs = [0, m + 1, M]
    h0 = synthetic.activations(r, M, TINY["hidden"])
    qn = np.concatenate([synthetic.logits_and_draft_probs(r, m, TINY["vocab"])[1] for _ in range(B)])
    dn = synthetic.sample_drafts(r, qn)
    un = synthetic.accept_uniforms(r, M)
    q, d, u = (torch.from_numpy(a).cuda() for a in (qn, dn, un))
    ref = _round(lib, model, offs, dev_bf16(h0), 1.0, q=q, draft=d, u=u)
    hidden, h_init = dev_bf16(h0), dev_bf16(h0)
    logits = torch.empty((M, TINY["vocab"]), dtype=torch.float32, device="cuda")
    out_len = torch.zeros(B, dtype=torch.int32).pin_memory()
    out_tokens = torch.full((M,), -1, dtype=torch.int32).pin_memory()
    ws = lib.workspace(lib.round_workspace_bytes(model, M))
    lib.verify_round(model, offs, hidden, 1.0, logits, out_len, out_tokens, ws, q=q, draft=d, u=u)
    torch.cuda.synchronize()
    assert (out_len.numpy() == ref[2]).all()
    for b in range(B):  # each request's committed tokens (entries past out_len are untouched)
        n = int(ref[2][b])
        assert (out_tokens.numpy()[offs[b]:offs[b] + n] == ref[3][offs[b]:offs[b] + n]).all()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s), torch.cuda.graph(g, stream=s):
        hidden.copy_(h_init)
        lib.verify_round(model, offs, hidden, 1.0, logits, out_len, out_tokens, ws, q=q, draft=d, u=u, stream=s)
    torch.cuda.synchronize()
    out_len.zero_()
    out_tokens.fill_(-1)
    g.replay()
    torch.cuda.synchronize()
    assert (out_len.numpy() == ref[2]).all()
    for b in range(B):
        n = int(ref[2][b])
        assert (out_tokens.numpy()[offs[b]:offs[b] + n] == ref[3][offs[b]:offs[b] + n]).all()
    assert lib.device_error() == 0

def _unpack_host(packed, N, K, bits):
    """Canonical (codes bytes [N, K*bits/8], scales, biases) read back from a unit-packed buffer,
    following the layout sv_qmm_pack documents: per (tile, chunk) unit, 128-byte pieces x 64 rows
    with 16-byte chunk c of row r at c ^ (r & 7), then 64 x 8 scales, then 64 x 8 biases."""
    rb = 512 * bits // 8
    wbytes, sb = 64 * rb, 64 * 8 * 2
    unit = wbytes + 2 * sb
    tiles, upt = (N + 63) // 64, K // 512
    buf = packed.cpu().numpy()
    codes = np.zeros((tiles * 64, K * bits // 8), np.uint8)
    sc = np.zeros((tiles * 64, K // 64), np.uint16)
    bi = np.zeros((tiles * 64, K // 64), np.uint16)
    for u in range(tiles * upt):
        t, kc = divmod(u, upt)
        blk = buf[u * unit:(u + 1) * unit]
        for r in range(64):
            for j in range(rb // 16):
                piece, c = divmod(j, 8)
                off = piece * 8192 + r * 128 + ((c ^ (r & 7)) << 4)
                codes[t * 64 + r, kc * rb + 16 * j: kc * rb + 16 * j + 16] = blk[off:off + 16]
        sc[t * 64:(t + 1) * 64, kc * 8:(kc + 1) * 8] = blk[wbytes:wbytes + sb].view(np.uint16).reshape(64, 8)
        bi[t * 64:(t + 1) * 64, kc * 8:(kc + 1) * 8] = blk[wbytes + sb:].view(np.uint16).reshape(64, 8)
    return codes, sc, bi


@pytest.mark.parametrize("bits,N", [(8, 1000), (4, 1024), (2, 1000)])
def test_pack_layout_round_trips(lib, bits, N):
    """The packed buffer holds exactly the canonical bytes in the documented order, zero rows past N."""
    r = synthetic.rng(1480 + bits)
    K = 1024
    w = _model.to_device(synthetic.quant_weight(r, N, K, bits, synthetic.LARGE_8BIT))
    packed = lib.pack(w)
    torch.cuda.synchronize()
    assert packed.numel() == lib.lib.sv_qmm_pack_bytes(N, K, bits) == ((N + 63) // 64) * 64 * K * (bits / 8 + 4 / 64)
    codes, sc, bi = _unpack_host(packed, N, K, bits)
    assert np.array_equal(codes[:N], w["wq"].cpu().numpy().view(np.uint8).reshape(N, -1))
    assert np.array_equal(sc[:N], w["scales"].cpu().numpy().view(np.uint16))
    assert np.array_equal(bi[:N], w["biases"].cpu().numpy().view(np.uint16))
    assert not codes[N:].any() and not sc[N:].any() and not bi[N:].any()


@pytest.mark.parametrize("bits", [2, 4, 8])
def test_packed_round_is_bitwise_the_canonical_round(lib, bits):
    layers, head = _model.host_model(1490 + bits, 2, bits=bits, stats={2: synthetic.TINY_2BIT, 4: synthetic.TINY_4BIT,
                                                                      8: synthetic.LARGE_8BIT}[bits], **TINY)
    dl, dh = _model.device_layers(layers), _model.to_device(head)
    canon = lib.make_model(dl, dh, TINY["hidden"], TINY["q_dim"], TINY["inter"], TINY["vocab"], bits)
    pl = [{k: dict(v, packed=lib.pack(v)) for k, v in layer.items()} for layer in dl]
    ph = dict(dh, packed=lib.pack(dh))
    packed = lib.make_model(pl, ph, TINY["hidden"], TINY["q_dim"], TINY["inter"], TINY["vocab"], bits)
    r = synthetic.rng(1495)
    m = 7
    h0 = dev_bf16(synthetic.activations(r, m + 1, TINY["hidden"]))
    _, z_q = synthetic.logits_and_draft_probs(r, m, TINY["vocab"])
    q = torch.from_numpy(z_q).cuda()
    draft = torch.from_numpy(synthetic.sample_drafts(r, z_q)).cuda()
    u = torch.from_numpy(synthetic.accept_uniforms(r, m + 1)).cuda()
    for T in (0.0, 0.7):
        a = _round(lib, canon, [0, m + 1], h0, T, q=q if T else None, draft=draft, u=u if T else None)
        b = _round(lib, packed, [0, m + 1], h0, T, q=q if T else None, draft=draft, u=u if T else None)
        assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
        assert np.array_equal(a[2], b[2]) and np.array_equal(a[3], b[3])
    assert lib.device_error() == 0


def test_round_refuses_a_plan_built_for_another_model(lib):
    layers, head = _model.host_model(1450, 1, bits=4, stats=synthetic.TINY_4BIT, **TINY)
    dl, dh = _model.device_layers(layers), _model.to_device(head)
    a = lib.make_model(dl, dh, TINY["hidden"], TINY["q_dim"], TINY["inter"], TINY["vocab"], 4)
    dh2 = _model.to_device(head)                     # same values, other device pointers
    b = lib.make_model(dl, dh2, TINY["hidden"], TINY["q_dim"], TINY["inter"], TINY["vocab"], 4)
    b.plan = a.plan
    h0 = dev_bf16(synthetic.activations(synthetic.rng(1451), 1, TINY["hidden"]))
    with pytest.raises(Exception, match="plan"):
        _round(lib, b, [0, 1], h0, 0.0, draft=torch.zeros(1, dtype=torch.int32, device="cuda"))
    _round(lib, a, [0, 1], h0, 0.0, draft=torch.zeros(1, dtype=torch.int32, device="cuda"))
    assert lib.device_error() == 0


QWEN8B = dict(hidden=4096, q_dim=4096, kv_dim=1024, inter=12288, vocab=151936)


@pytest.fixture(scope="module")
def model_8b():
    layers, head = _model.device_random_model(1500, 36, bits=8, stats=synthetic.LARGE_8BIT, **QWEN8B)
    yield layers, head
    del layers, head
    torch.cuda.empty_cache()


@pytest.mark.parametrize("M,T", [(8, 0.7), (16, 0.0), (1, 0.7)])
def test_qwen3_8b_round_per_layer_and_head(lib, model_8b, M, T):
    """Full 36-layer 8-bit round, the benchmark's launch configuration: each checked
    layer is compared with the oracle applied to the GPU's own input of that layer."""
    layers, head = model_8b
    r = synthetic.rng(1600 + M)
    h0 = dev_bf16(synthetic.activations(r, M, QWEN8B["hidden"]))
    m = M - 1
    q = u = None
    if T > 0 and m:
        _, qn = synthetic.logits_and_draft_probs(r, m, QWEN8B["vocab"])
        q = torch.from_numpy(qn).cuda()
    if T > 0:
        u = torch.from_numpy(synthetic.accept_uniforms(r, m + 1)).cuda()
    draft = torch.from_numpy(r.integers(0, QWEN8B["vocab"], m).astype(np.int32)).cuda()

    def run(depth):
        model = lib.make_model(layers[:depth], head, QWEN8B["hidden"], QWEN8B["q_dim"], QWEN8B["inter"],
                               QWEN8B["vocab"], 8)
        return _round(lib, model, [0, M], h0, T, q=q, draft=draft, u=u)

    for depth in (1, 18, 36):
        before = host_bf16_bits(run(depth - 1)[0]) if depth > 1 else host_bf16_bits(h0)
        after, logits, n, toks = run(depth)
        lay = _model.split_device_layer(layers[depth - 1], QWEN8B["q_dim"], QWEN8B["kv_dim"], QWEN8B["inter"])
        want = chain.layer_forward(before, lay)
        # the hidden state is rounded to bf16 twice in a layer (h + o, then + down)
        assert_close_bf16(host_f32_of_bf16(after), quant.bf16_bits_to_f32(want), what="layer %d" % depth, ulps=2)
    # vocab head on sampled rows, from the GPU's final hidden state
    lg = logits.cpu().numpy()
    rows = np.unique(np.concatenate([r.choice(QWEN8B["vocab"], 2048, replace=False), np.argmax(lg, axis=1)]))
    hw = _model.host_copy(head)
    sub = {"wq": hw["wq"][rows], "scales": hw["scales"][rows], "biases": hw["biases"][rows], "K": QWEN8B["hidden"],
           "bits": 8}
    want = chain.normed_f64(sub, host_bf16_bits(after)).astype(np.float32)   # head of the final RMSNorm
    assert_close_rms(lg[:, rows], want, what="head rows")
    # accept on identical logits
    dn = draft.cpu().numpy()
    if T > 0:
        det = oa.sampled_accept_detail(lg, q.cpu().numpy() if q is not None else np.zeros((0, lg.shape[1]), np.float32),
                                       dn, T, u.cpu().numpy())
        want_acc = (det["out_len"], det["tokens"])
    else:
        want_acc = tuple(oa.greedy_accept(lg, dn))
    assert (int(n[0]), toks[:n[0]].tolist()) == want_acc
    assert lib.device_error() == 0


def _check_round_layers(lib, layers, head, shape, offs, h0, T, depths, q=None, draft=None, u=None, bits=8):
    """Run the round at each prefix depth and compare the checked layers (given the
    GPU's own input of that layer) and the head's sampled rows with the oracle."""
    r = synthetic.rng(sum(depths))

    def run(depth):
        model = lib.make_model(layers[:depth], head, shape["hidden"], shape["q_dim"], shape["inter"], shape["vocab"],
                               bits)
        return _round(lib, model, offs, h0, T, q=q, draft=draft, u=u)

    for depth in depths:
        before = host_bf16_bits(run(depth - 1)[0]) if depth > 1 else host_bf16_bits(h0)
        after, logits, n, toks = run(depth)
        lay = _model.split_device_layer(layers[depth - 1], shape["q_dim"], shape["kv_dim"], shape["inter"])
        want = chain.layer_forward(before, lay)
        # the hidden state is rounded to bf16 twice in a layer (h + o, then + down)
        assert_close_bf16(host_f32_of_bf16(after), quant.bf16_bits_to_f32(want), what="layer %d" % depth, ulps=2)
    lg = logits.cpu().numpy()
    rows = np.unique(np.concatenate([r.choice(shape["vocab"], 2048, replace=False), np.argmax(lg, axis=1)]))
    hw = _model.host_copy(head)
    sub = {"wq": hw["wq"][rows], "scales": hw["scales"][rows], "biases": hw["biases"][rows], "K": shape["hidden"],
           "bits": bits}
    assert_close_rms(lg[:, rows], chain.normed_f64(sub, host_bf16_bits(after)).astype(np.float32), what="head rows")
    return lg, n, toks


QWEN4B = dict(hidden=2560, q_dim=4096, kv_dim=1024, inter=9728, vocab=151936)


@pytest.mark.parametrize("M,T", [(8, 0.0), (32, 0.7)])
def test_qwen3_4b_shaped_4bit_round(lib, M, T):
    """4B-shaped 4-bit target (hidden 2560, q 4096, kv 1024, inter 9728, the full
    151936-row head): a 3-layer prefix model, every layer and the head checked."""
    layers, head = _model.device_random_model(2100 + M, 3, bits=4, stats=synthetic.LARGE_8BIT, **QWEN4B)
    r = synthetic.rng(2101 + M)
    m = M - 1
    h0 = dev_bf16(synthetic.activations(r, M, QWEN4B["hidden"]))
    q = u = None
    if T > 0:
        _, qn = synthetic.logits_and_draft_probs(r, m, QWEN4B["vocab"])
        q = torch.from_numpy(qn).cuda()
        u = torch.from_numpy(synthetic.accept_uniforms(r, M)).cuda()
    draft = torch.from_numpy(r.integers(0, QWEN4B["vocab"], m).astype(np.int32)).cuda()
    lg, n, toks = _check_round_layers(lib, layers, head, QWEN4B, [0, M], h0, T, (1, 2, 3), q=q, draft=draft, u=u,
                                      bits=4)
    dn = draft.cpu().numpy()
    if T > 0:
        det = oa.sampled_accept_detail(lg, q.cpu().numpy(), dn, T, u.cpu().numpy())
        want = (det["out_len"], det["tokens"])
    else:
        want = tuple(oa.greedy_accept(lg, dn))
    assert (int(n[0]), toks[:n[0]].tolist()) == want
    assert lib.device_error() == 0


QWEN27B = dict(hidden=5120, q_dim=6144, kv_dim=1024, inter=17408, vocab=151936)


def test_27b_class_64_layer_batched_round(lib):
    """27B-class 8-bit shapes in one 64-layer launch (257 phases), B = 4 requests x
    (1 + 7) rows = 32 rows, T = 1.0, each request's uniforms from its own Philox
    stream; layers 1, 32 and 64 and the head against the oracle, then each
    request's accept on the GPU's logits."""
    layers, head = _model.device_random_model(2700, 64, bits=8, stats=synthetic.LARGE_8BIT, **QWEN27B)
    r = synthetic.rng(2701)
    B, rows = 4, 8
    M, m = B * rows, rows - 1
    offs = [b * rows for b in range(B + 1)]
    h0 = dev_bf16(synthetic.activations(r, M, QWEN27B["hidden"]))
    _, qn = synthetic.logits_and_draft_probs(r, B * m, QWEN27B["vocab"])
    q = torch.from_numpy(qn).cuda()
    u = torch.cat([lib.philox_uniforms(2702, b, 0, rows) for b in range(B)])
    draft = torch.from_numpy(r.integers(0, QWEN27B["vocab"], B * m).astype(np.int32)).cuda()
    lg, n, toks = _check_round_layers(lib, layers, head, QWEN27B, offs, h0, 1.0, (1, 32, 64), q=q, draft=draft, u=u)
    uh, dn, qh = u.cpu().numpy(), draft.cpu().numpy(), q.cpu().numpy()
    for b in range(B):
        det = oa.sampled_accept_detail(lg[offs[b]:offs[b + 1]], qh[b * m:(b + 1) * m], dn[b * m:(b + 1) * m], 1.0,
                                       uh[offs[b]:offs[b + 1]])
        got = (int(n[b]), toks[offs[b]:offs[b] + n[b]].tolist())
        assert got == (det["out_len"], det["tokens"]) or _near_tie(det, uh[offs[b]:offs[b + 1]]), b
    del layers, head
    torch.cuda.empty_cache()
    assert lib.device_error() == 0


def _near_tie(det, u):
    for i, rr in enumerate(det["ratios"]):
        if np.isfinite(rr) and abs(float(u[i]) - rr) < 1e-6:
            return True
    return bool(np.min(np.abs(det["cdf"] - det["theta"])) < 1e-6 * det["Z"])
