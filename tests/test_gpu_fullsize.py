"""Full-size workloads on the GPU, checked against the oracle on sampled outputs.

The inputs are generated on the device by the same counter-based generator as
the numpy version; the sampled rows the oracle needs are regenerated with numpy
and must be bit-identical to the device rows.  Every step of the layer is
row-independent (and the backward weight is independent per Hadamard block
along K), so the oracle recomputes exactly the sampled rows, blocks and output
entries.  Sizes are the full workload sizes and the calls are the ones the
benchmark times.
"""
import numpy as np
import pytest

import oracle
import synth
from helpers import (REL_FRO_BF16, REL_FRO_ORACLE, bits_of, check_codes, check_dequant_elementwise, check_scales,
                     codes_of, f64, rel_fro)

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import int8_rotated_quantized_gb300 as cr  # noqa: E402
import synth.gpu as sg  # noqa: E402

N_SAMPLE = 48


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    cr._build.build()
    cr.lib()


def _rows(rng, n, count=N_SAMPLE):
    return np.sort(rng.choice(n, size=min(count, n), replace=False))


def _act_rows(wl, rows, K, stream=synth.STREAM_X):
    return np.concatenate([synth.activations_bf16(0, 1, K, wl["x_outliers"], wl["x_factor"], row0=int(r),
                                                  stream=stream) for r in rows])


def _normal_rows(stream, rows, cols, sigma):
    return np.concatenate([synth.normal_bf16(0, stream, 1, cols, sigma, row0=int(r)) for r in rows])


def _oracle_weight(W_gpu, Wq, sw, b):
    """The oracle's quantization of the whole weight (its input: the bits of the shared
    seeded generator), checked against the GPU's, and uploaded so that the GPU's
    backward runs on exactly the codes the oracle's reference uses."""
    w_np = bits_of(W_gpu)
    wq_ref, sw_ref = oracle.quantize_rows_bf16(w_np, b)
    check_codes(codes_of(Wq), wq_ref, f64(w_np), b, "weight codes (all rows)")
    check_scales(sw.cpu().numpy(), sw_ref, "weight scales (all rows)")
    wq_dev = torch.from_numpy(wq_ref).cuda()
    sw_dev = torch.from_numpy(sw_ref).cuda()
    return wq_ref, sw_ref, wq_dev, sw_dev


def _check_fwd(wl, x_gpu, W_gpu, Wq, sw, y, rng):
    M, K = x_gpu.shape
    N = W_gpu.shape[0]
    b = wl["block"]
    ms, ns = _rows(rng, M), _rows(rng, N)
    x_rows = _act_rows(wl, ms, K)
    w_rows = _normal_rows(synth.STREAM_W, ns, K, wl["w_sigma"])
    assert np.array_equal(bits_of(x_gpu[torch.from_numpy(ms).cuda()]), x_rows), "device generator differs"
    assert np.array_equal(bits_of(W_gpu[torch.from_numpy(ns).cuda()]), w_rows), "device generator differs"
    wq_ref, sw_ref = oracle.quantize_rows_bf16(w_rows, b)
    check_codes(codes_of(Wq[torch.from_numpy(ns).cuda()]), wq_ref, f64(w_rows), b, "weight codes")
    check_scales(sw.cpu().numpy()[ns], sw_ref, "weight scales")
    y_ref, xq_ref, _ = oracle.linear_fwd(x_rows, wq_ref, sw_ref, b)
    y_s = bits_of(y[torch.from_numpy(ms).cuda()][:, torch.from_numpy(ns).cuda()])
    assert rel_fro(f64(y_s), f64(y_ref)) <= REL_FRO_ORACLE
    assert rel_fro(f64(y_s), f64(x_rows) @ f64(w_rows).T) <= REL_FRO_BF16
    # element by element on the sampled outputs whose activation and weight code rows agree
    # with the oracle's (the forward's own quantizer kernel gives the GPU's activation codes)
    xq, _ = cr.convrot_quantize_activation(x_gpu, b)
    rows_ok = np.all(codes_of(xq[torch.from_numpy(ms).cuda()]) == xq_ref, axis=1)
    cols_ok = np.all(codes_of(Wq[torch.from_numpy(ns).cuda()]) == wq_ref, axis=1)
    mask = rows_ok[:, None] & cols_ok[None, :]
    assert mask.mean() > 0.9
    check_dequant_elementwise(y_s, y_ref, mask=mask, what="full-size forward (sampled)")
    del xq


def test_img1024_forward_full_size():
    wl = synth.WORKLOADS["img1024"]
    M, K, N, b = wl["M"], wl["K"], wl["N"], wl["block"]
    x = sg.activations_bf16(0, M, K, wl["x_outliers"], wl["x_factor"], "cuda")
    W = sg.normal_bf16(0, synth.STREAM_W, N, K, wl["w_sigma"], "cuda")
    Wq, sw = cr.convrot_quantize_weight(W, b)
    y = cr.convrot_linear_fwd(x, Wq, sw, b)
    assert cr.convrot_get_error() == cr.OK
    _check_fwd(wl, x, W, Wq, sw, y, np.random.default_rng(1))
    # activation codes of sampled rows
    xq, sx = cr.convrot_quantize_activation(x, b)
    ms = _rows(np.random.default_rng(2), M)
    x_rows = _act_rows(wl, ms, K)
    q_ref, s_ref = oracle.quantize_rows_bf16(x_rows, b)
    check_codes(codes_of(xq[torch.from_numpy(ms).cuda()]), q_ref, f64(x_rows), b, "activation codes")
    check_scales(sx.cpu().numpy()[ms], s_ref, "activation scales")


def test_qkv_lora_merge_and_forward_full_size():
    wl = synth.WORKLOADS["qkv_lora"]
    M, K, N, b = wl["M"], wl["K"], wl["N"], wl["block"]
    r, alpha, scale = wl["lora_rank"], wl["lora_alpha"], wl["lora_scale"]
    W = sg.normal_bf16(0, synth.STREAM_W, N, K, wl["w_sigma"], "cuda")
    A, B = sg.lora_pair(0, N, K, r, wl["lora_sigma"], "cuda")
    Wq, sw = cr.convrot_quantize_weight(W, b, A, B, alpha, scale)
    x = sg.activations_bf16(0, M, K, wl["x_outliers"], wl["x_factor"], "cuda")
    y = cr.convrot_linear_fwd(x, Wq, sw, b)
    assert cr.convrot_get_error() == cr.OK
    rng = np.random.default_rng(3)
    ns, ms = _rows(rng, N), _rows(rng, M)
    A_np, B_np = synth.lora_pair(0, N, K, r, wl["lora_sigma"])
    assert np.array_equal(A.cpu().numpy(), A_np) and np.array_equal(B.cpu().numpy(), B_np)
    w_rows = _normal_rows(synth.STREAM_W, ns, K, wl["w_sigma"])
    assert np.array_equal(bits_of(W[torch.from_numpy(ns).cuda()]), w_rows)
    wq_ref, sw_ref = oracle.quantize_weight(w_rows, b, A_np, B_np[ns], alpha, scale)
    merged = oracle.lora_merge(w_rows, A_np, B_np[ns], alpha, scale)
    check_codes(codes_of(Wq[torch.from_numpy(ns).cuda()]), wq_ref, f64(merged), b, "merged weight codes")
    check_scales(sw.cpu().numpy()[ns], sw_ref, "merged weight scales")
    x_rows = _act_rows(wl, ms, K)
    y_ref, _, _ = oracle.linear_fwd(x_rows, wq_ref, sw_ref, b)
    y_s = bits_of(y[torch.from_numpy(ms).cuda()][:, torch.from_numpy(ns).cuda()])
    assert rel_fro(f64(y_s), f64(y_ref)) <= REL_FRO_ORACLE
    assert rel_fro(f64(y_s), f64(x_rows) @ f64(merged).T) <= REL_FRO_BF16


def test_qkv_lora_bypass_forward_full_size():
    wl = synth.WORKLOADS["qkv_lora"]
    M, K, N, b = wl["M"], wl["K"], wl["N"], wl["block"]
    r, alpha, scale = wl["lora_rank"], wl["lora_alpha"], wl["lora_scale"]
    W = sg.normal_bf16(0, synth.STREAM_W, N, K, wl["w_sigma"], "cuda")
    A, B = sg.lora_pair(0, N, K, r, wl["lora_sigma"], "cuda")
    Wq, sw = cr.convrot_quantize_weight(W, b)
    x = sg.activations_bf16(0, M, K, wl["x_outliers"], wl["x_factor"], "cuda")
    y = cr.convrot_linear_fwd_lora(x, Wq, sw, b, A, B, alpha, scale)
    assert cr.convrot_get_error() == cr.OK
    rng = np.random.default_rng(7)
    ns, ms = _rows(rng, N), _rows(rng, M)
    A_np, B_np = synth.lora_pair(0, N, K, r, wl["lora_sigma"])
    x_rows = _act_rows(wl, ms, K)
    assert np.array_equal(bits_of(x[torch.from_numpy(ms).cuda()]), x_rows)
    w_rows = _normal_rows(synth.STREAM_W, ns, K, wl["w_sigma"])
    wq_s, sw_s = oracle.quantize_rows_bf16(w_rows, b)
    check_codes(codes_of(Wq[torch.from_numpy(ns).cuda()]), wq_s, f64(w_rows), b, "weight codes")
    check_scales(sw.cpu().numpy()[ns], sw_s, "weight scales")
    ref = oracle.linear_fwd_lora(x_rows, wq_s, sw_s, b, A_np, B_np[ns], alpha, scale)
    got = bits_of(y[torch.from_numpy(ms).cuda()][:, torch.from_numpy(ns).cuda()])
    assert rel_fro(f64(got), f64(ref)) <= REL_FRO_ORACLE
    assert np.mean(got == ref) > 0.9
    merged = oracle.lora_merge(w_rows, A_np, B_np[ns], alpha, scale)
    assert rel_fro(f64(got), f64(x_rows) @ f64(merged).T) <= REL_FRO_BF16


def test_train20k_forward_and_backward_full_size():
    wl = synth.WORKLOADS["train20k"]
    M, K, N, b = wl["M"], wl["K"], wl["N"], wl["block"]
    x = sg.activations_bf16(0, M, K, wl["x_outliers"], wl["x_factor"], "cuda")
    W = sg.normal_bf16(0, synth.STREAM_W, N, K, wl["w_sigma"], "cuda")
    Wq, sw = cr.convrot_quantize_weight(W, b)
    y = cr.convrot_linear_fwd(x, Wq, sw, b)
    rng = np.random.default_rng(4)
    _check_fwd(wl, x, W, Wq, sw, y, rng)
    del y
    # backward: the prepared weight on two Hadamard blocks along K, then grad_x, on the
    # oracle's weight codes (checked against the GPU's on every row)
    wq_np, sw_np, Wq_o, sw_o = _oracle_weight(W, Wq, sw, b)
    WtQ, swt = cr.convrot_prepare_bwd_weight(Wq_o, sw_o, b)
    dY = sg.normal_bf16(0, synth.STREAM_DY, M, N, wl["dy_sigma"], "cuda")
    dX = cr.convrot_linear_bwd_x(dY, WtQ, swt, b)
    assert cr.convrot_get_error() == cr.OK
    kblocks = np.sort(rng.choice(K // b, size=2, replace=False))
    ks = np.concatenate([np.arange(kb * b, (kb + 1) * b) for kb in kblocks])
    wtq_ref = np.empty((len(ks), N), dtype=np.int8)
    swt_ref = np.empty(len(ks), dtype=np.float32)
    for i, kb in enumerate(kblocks):
        q, s = oracle.prepare_bwd_weight(np.ascontiguousarray(wq_np[:, kb * b:(kb + 1) * b]), sw_np, b)
        wtq_ref[i * b:(i + 1) * b], swt_ref[i * b:(i + 1) * b] = q, s
    w_eff_t = np.concatenate([oracle.rotate_rows(sw_np[:, None].astype(np.float64) *
                                                 wq_np[:, kb * b:(kb + 1) * b], b).T for kb in kblocks])
    check_codes(codes_of(WtQ[torch.from_numpy(ks).cuda()]), wtq_ref, w_eff_t, b, "backward weight codes")
    check_scales(swt.cpu().numpy()[ks], swt_ref, "backward weight scales")
    ms = _rows(rng, M)
    dy_rows = _normal_rows(synth.STREAM_DY, ms, N, wl["dy_sigma"])
    assert np.array_equal(bits_of(dY[torch.from_numpy(ms).cuda()]), dy_rows)
    dx_ref, _, _ = oracle.linear_bwd_x(dy_rows, wtq_ref, swt_ref, b)
    dx_s = bits_of(dX[torch.from_numpy(ms).cuda()][:, torch.from_numpy(ks).cuda()])
    assert rel_fro(f64(dx_s), f64(dx_ref)) <= REL_FRO_ORACLE
    w_rows_k = bits_of(W[:, torch.from_numpy(ks).cuda()])
    assert rel_fro(f64(dx_s), f64(dy_rows) @ f64(w_rows_k)) <= REL_FRO_BF16


def test_dequant_weight_t_on_l2_resident_codes_full_size():
    """The transient transpose of the bf16 backward, made from codes the quantizer
    has just written (resident in L2, so the copies into the kernel's int8 ring
    land fast), and twice more after touching the codes again: every element of
    every call equals the oracle.  (A stage handed back to the copy engine
    before its loads were performed showed up only in this regime.)"""
    wl = synth.WORKLOADS["train20k"]
    K, N, b = wl["K"], wl["N"], wl["block"]
    W = sg.normal_bf16(0, synth.STREAM_W, N, K, wl["w_sigma"], "cuda")
    Wq, sw = cr.convrot_quantize_weight(W, b)
    Ts = [cr.convrot_dequant_weight_t(Wq, sw, b)]
    for _ in range(2):
        Wq.add_(0)  # the codes back into L2
        Ts.append(cr.convrot_dequant_weight_t(Wq, sw, b))
    assert cr.convrot_get_error() == cr.OK
    wq_np, sw_np = Wq.cpu().numpy(), sw.cpu().numpy()
    Tb = [T.view(torch.int16).cpu().numpy().view(np.uint16) for T in Ts]
    for kb in range(K // b):
        ref = oracle.dequant_weight_t(np.ascontiguousarray(wq_np[:, kb * b:(kb + 1) * b]), sw_np, b)
        for T in Tb:
            np.testing.assert_array_equal(T[kb * b:(kb + 1) * b], ref)


def test_train20k_bf16_backward_full_size():
    wl = synth.WORKLOADS["train20k"]
    M, K, N, b = wl["M"], wl["K"], wl["N"], wl["block"]
    W = sg.normal_bf16(0, synth.STREAM_W, N, K, wl["w_sigma"], "cuda")
    Wq, sw = cr.convrot_quantize_weight(W, b)
    wq_np, sw_np, Wq_o, sw_o = _oracle_weight(W, Wq, sw, b)
    dY = sg.normal_bf16(0, synth.STREAM_DY, M, N, wl["dy_sigma"], "cuda")
    ws = torch.empty(cr.convrot_bwd_x_bf16_workspace_bytes(N, K), dtype=torch.uint8, device="cuda")
    dX = cr.convrot_linear_bwd_x_bf16(dY, Wq_o, sw_o, b, workspace=ws)
    assert cr.convrot_get_error() == cr.OK
    rng = np.random.default_rng(6)
    kblocks = np.sort(rng.choice(K // b, size=2, replace=False))
    ks = np.concatenate([np.arange(kb * b, (kb + 1) * b) for kb in kblocks])
    weff_ref = np.concatenate([oracle.dequant_weight_t(np.ascontiguousarray(wq_np[:, kb * b:(kb + 1) * b]), sw_np, b)
                               for kb in kblocks])                      # [len(ks), N]
    weff_dev = ws[:K * N * 2].view(torch.int16).view(K, N)[torch.from_numpy(ks).cuda()].cpu().numpy().view(np.uint16)
    np.testing.assert_array_equal(weff_dev, weff_ref)
    ms = _rows(rng, M)
    dy_rows = _normal_rows(synth.STREAM_DY, ms, N, wl["dy_sigma"])
    assert np.array_equal(bits_of(dY[torch.from_numpy(ms).cuda()]), dy_rows)
    dx_ref = oracle.gemm_bf16(dy_rows, weff_ref)
    dx_s = bits_of(dX[torch.from_numpy(ms).cuda()][:, torch.from_numpy(ks).cuda()])
    g, r = f64(dx_s), f64(dx_ref)
    # one bf16 step, plus the fp32 accumulation of N terms near zero (see the parity tests)
    assert np.all(np.abs(g - r) <= np.abs(r) * 2.0 ** -7 + 64 * 2.0 ** -24 * np.sqrt(N) * np.sqrt(np.mean(r * r)))
    assert np.mean(dx_s == dx_ref) > 0.98
    w_cols = bits_of(W[:, torch.from_numpy(ks).cuda()])
    assert rel_fro(g, f64(dy_rows) @ f64(w_cols)) <= REL_FRO_BF16


def test_train20k_int8_backward_second_reading_full_size():
    wl = synth.WORKLOADS["train20k"]
    M, K, N, b = wl["M"], wl["K"], wl["N"], wl["block"]
    W = sg.normal_bf16(0, synth.STREAM_W, N, K, wl["w_sigma"], "cuda")
    Wq, sw = cr.convrot_quantize_weight(W, b)
    wq_np, sw_np, Wq_o, sw_o = _oracle_weight(W, Wq, sw, b)
    dY = sg.normal_bf16(0, synth.STREAM_DY, M, N, wl["dy_sigma"], "cuda")
    ws = torch.empty(cr.convrot_bwd_x_r2_workspace_bytes(M, N, K), dtype=torch.uint8, device="cuda")
    dX = cr.convrot_linear_bwd_x_r2(dY, Wq_o, sw_o, b, workspace=ws)
    assert cr.convrot_get_error() == cr.OK
    rng = np.random.default_rng(9)
    ms = _rows(rng, M, 16)
    dy_rows = _normal_rows(synth.STREAM_DY, ms, N, wl["dy_sigma"])
    assert np.array_equal(bits_of(dY[torch.from_numpy(ms).cuda()]), dy_rows)
    dx_ref, dq_ref, sd_ref = oracle.linear_bwd_x_r2(dy_rows, wq_np, sw_np, b)
    # the unrotated codes and the row scales are decided in the same fp32 arithmetic: identical
    dq = ws[:M * N * 2].view(torch.float16).view(M, N)[torch.from_numpy(ms).cuda()]
    np.testing.assert_array_equal(codes_of(dq), dq_ref)
    off = (M * N * 2 + 255) // 256 * 256
    np.testing.assert_array_equal(ws[off:off + 4 * M].view(torch.float32).cpu().numpy()[ms], sd_ref)
    got = bits_of(dX[torch.from_numpy(ms).cuda()])
    g, r = f64(got), f64(dx_ref)
    # one bf16 step, plus an allowance for the fp32 scaling and rotation near zero (as the parity tests)
    assert np.all(np.abs(g - r) <= np.abs(r) * 2.0 ** -7 + 64 * 2.0 ** -24 * np.sqrt(K) * np.sqrt(np.mean(r * r)))
    assert np.mean(got == dx_ref) > 0.98
    assert rel_fro(g, f64(dy_rows) @ f64(bits_of(W))) <= REL_FRO_BF16


def test_embed_table_and_lookup_full_size():
    wl = synth.WORKLOADS["embed"]
    V, D, b, n = wl["V"], wl["D"], wl["block"], wl["n_ids"]
    T = sg.normal_bf16(0, synth.STREAM_TABLE, V, D, wl["table_sigma"], "cuda")
    Eq = torch.empty((V, D), dtype=torch.int8, device="cuda")
    se = torch.empty((V,), dtype=torch.float32, device="cuda")
    slab = 31000
    for r0 in range(0, V, slab):
        r1 = min(V, r0 + slab)
        cr.convrot_quantize_weight(T[r0:r1], b, Wq=Eq[r0:r1], scale_w=se[r0:r1])
    ids = sg.token_ids(0, n, V, "cuda", set_index=0)
    out = cr.convrot_embedding_lookup(ids, Eq, se, b)
    assert cr.convrot_get_error() == cr.OK
    rng = np.random.default_rng(5)
    vs = _rows(rng, V)
    t_rows = _normal_rows(synth.STREAM_TABLE, vs, D, wl["table_sigma"])
    assert np.array_equal(bits_of(T[torch.from_numpy(vs).cuda()]), t_rows)
    q_ref, s_ref = oracle.quantize_rows_bf16(t_rows, b)
    check_codes(codes_of(Eq[torch.from_numpy(vs).cuda()]), q_ref, f64(t_rows), b, "table codes")
    check_scales(se.cpu().numpy()[vs], s_ref, "table scales")
    ids_np = synth.token_ids(0, n, V, set_index=0)
    assert np.array_equal(ids.cpu().numpy(), ids_np)
    ts = _rows(rng, n)
    sel = ids_np[ts]
    t_sel = _normal_rows(synth.STREAM_TABLE, sel, D, wl["table_sigma"])
    q_sel, s_sel = oracle.quantize_rows_bf16(t_sel, b)
    ref, bad = oracle.embedding_lookup(np.arange(len(sel), dtype=np.int64), q_sel, s_sel, b)
    assert bad == 0
    got = bits_of(out[torch.from_numpy(ts).cuda()])
    assert rel_fro(f64(got), f64(ref)) <= REL_FRO_ORACLE
    assert rel_fro(f64(got), f64(t_sel)) < 2e-2
