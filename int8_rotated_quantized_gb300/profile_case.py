"""Runs one kernel of libconvrot on a fixed synthetic case, a few times, for
profilers (ncu) and quick timing.

    python -m int8_rotated_quantized_gb300.profile_case gemm --M 8192 --N 16384 --K 4096
    python -m int8_rotated_quantized_gb300.profile_case rotq --M 20480 --K 4096
    python -m int8_rotated_quantized_gb300.profile_case lookup --V 248000 --D 4096 --n 8192
    python -m int8_rotated_quantized_gb300.profile_case lora --N 12288 --K 4096
    python -m int8_rotated_quantized_gb300.profile_case prep --N 16384 --K 4096
    python -m int8_rotated_quantized_gb300.profile_case bwd_r2 --M 20480 --N 16384 --K 4096

Each case does one warm-up launch and `--reps` measured launches (CUDA events,
L2 flushed before each) and prints the median time.
"""
from __future__ import annotations

import argparse
import os
import statistics
import sys

import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import int8_rotated_quantized_gb300 as cr  # noqa: E402
import synth  # noqa: E402
import synth.gpu as sg  # noqa: E402


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("case", choices=["gemm", "gemm_w16", "gemm_bf16", "widen", "rotq", "lookup", "lora", "prep",
                                     "dequant", "wquant", "bwd_r2", "fwd_lora"])
    ap.add_argument("--M", type=int, default=8192)
    ap.add_argument("--N", type=int, default=16384)
    ap.add_argument("--K", type=int, default=4096)
    ap.add_argument("--V", type=int, default=248000)
    ap.add_argument("--D", type=int, default=4096)
    ap.add_argument("--n", type=int, default=8192)
    ap.add_argument("--block", type=int, default=128)
    ap.add_argument("--reps", type=int, default=3)
    a = ap.parse_args()
    cr._build.build()
    dev = torch.device("cuda", 0)
    b = a.block
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    if a.case == "gemm":
        x = sg.activations_bf16(0, a.M, a.K, 41, 30.0, dev)
        W = sg.normal_bf16(0, synth.STREAM_W, a.N, a.K, 0.02, dev)
        Wq, sw = cr.convrot_quantize_weight(W, b)
        xq, sx = cr.convrot_quantize_activation(x, b)
        y = torch.empty((a.M, a.N), dtype=torch.bfloat16, device=dev)
        fn = lambda i: cr.convrot_gemm_dequant(xq, sx, Wq, sw, None, y)  # noqa: E731
        work = 2.0 * a.M * a.N * a.K
        unit = "TOPS"
    elif a.case == "gemm_w16":
        x = sg.activations_bf16(0, a.M, a.K, 41, 30.0, dev)
        W = sg.normal_bf16(0, synth.STREAM_W, a.N, a.K, 0.02, dev)
        Wq, sw = cr.convrot_quantize_weight(W, b)
        W16 = cr.convrot_widen_codes(Wq)
        xq, sx = cr.convrot_quantize_activation(x, b)
        y = torch.empty((a.M, a.N), dtype=torch.bfloat16, device=dev)
        fn = lambda i: cr.convrot_gemm_dequant_w16(xq, sx, W16, sw, None, y)  # noqa: E731
        work = 2.0 * a.M * a.N * a.K
        unit = "TOPS"
    elif a.case == "widen":
        W = sg.normal_bf16(0, synth.STREAM_W, a.N, a.K, 0.02, dev)
        Wq, sw = cr.convrot_quantize_weight(W, b)
        W16 = torch.empty((a.N, a.K), dtype=torch.float16, device=dev)
        fn = lambda i: cr.convrot_widen_codes(Wq, W16)  # noqa: E731
        work = 3 * a.N * a.K
        unit = "GB/s"
    elif a.case == "gemm_bf16":
        A = sg.normal_bf16(0, synth.STREAM_DY, a.M, a.K, 1e-3, dev)
        B = sg.normal_bf16(0, synth.STREAM_W, a.N, a.K, 0.02, dev)
        y = torch.empty((a.M, a.N), dtype=torch.bfloat16, device=dev)
        fn = lambda i: cr.convrot_gemm_bf16(A, B, y)  # noqa: E731
        work = 2.0 * a.M * a.N * a.K
        unit = "TOPS"
    elif a.case == "rotq":
        x = sg.activations_bf16(0, a.M, a.K, 41, 30.0, dev)
        xq = torch.empty((a.M, a.K), dtype=torch.float16, device=dev)
        sx = torch.empty((a.M,), dtype=torch.float32, device=dev)
        fn = lambda i: cr.convrot_quantize_activation(x, b, xq, sx)  # noqa: E731
        work = a.M * a.K * 4 + a.M * 4
        unit = "GB/s"
    elif a.case == "wquant":
        W = sg.normal_bf16(0, synth.STREAM_W, a.N, a.K, 0.02, dev)
        Wq = torch.empty((a.N, a.K), dtype=torch.int8, device=dev)
        sw = torch.empty((a.N,), dtype=torch.float32, device=dev)
        fn = lambda i: cr.convrot_quantize_weight(W, b, Wq=Wq, scale_w=sw)  # noqa: E731
        work = a.N * a.K * 3 + a.N * 4
        unit = "GB/s"
    elif a.case == "lora":
        W = sg.normal_bf16(0, synth.STREAM_W, a.N, a.K, 0.02, dev)
        A, B = sg.lora_pair(0, a.N, a.K, 16, 0.01, dev)
        Wq = torch.empty((a.N, a.K), dtype=torch.int8, device=dev)
        sw = torch.empty((a.N,), dtype=torch.float32, device=dev)
        fn = lambda i: cr.convrot_quantize_weight(W, b, A, B, 16.0, 1.0, Wq, sw)  # noqa: E731
        work = a.N * a.K * 3 + a.N * 4 + 16 * a.K * 4 + a.N * 16 * 4
        unit = "GB/s"
    elif a.case == "prep":
        W = sg.normal_bf16(0, synth.STREAM_W, a.N, a.K, 0.02, dev)
        Wq, sw = cr.convrot_quantize_weight(W, b)
        WtQ = torch.empty((a.K, a.N), dtype=torch.int8, device=dev)
        swt = torch.empty((a.K,), dtype=torch.float32, device=dev)
        ws = torch.empty(cr.convrot_bwd_weight_workspace_bytes(a.N, a.K), dtype=torch.uint8, device=dev)
        fn = lambda i: cr.convrot_prepare_bwd_weight(Wq, sw, b, WtQ, swt, ws)  # noqa: E731
        work = 2 * a.N * a.K + 4 * (a.N + a.K)
        unit = "GB/s"
    elif a.case == "dequant":
        W = sg.normal_bf16(0, synth.STREAM_W, a.N, a.K, 0.02, dev)
        Wq, sw = cr.convrot_quantize_weight(W, b)
        T = torch.empty((a.K, a.N), dtype=torch.bfloat16, device=dev)
        fn = lambda i: cr.convrot_dequant_weight_t(Wq, sw, b, T)  # noqa: E731
        work = a.N * a.K + a.N * 4 + 2 * a.N * a.K
        unit = "GB/s"
    elif a.case == "bwd_r2":
        # --N out features (dY width), --K in features
        dY = sg.normal_bf16(0, synth.STREAM_DY, a.M, a.N, 1e-3, dev)
        W = sg.normal_bf16(0, synth.STREAM_W, a.N, a.K, 0.02, dev)
        Wq, sw = cr.convrot_quantize_weight(W, b)
        dX = torch.empty((a.M, a.K), dtype=torch.bfloat16, device=dev)
        ws = torch.empty(cr.convrot_bwd_x_r2_workspace_bytes(a.M, a.N, a.K), dtype=torch.uint8, device=dev)
        fn = lambda i: cr.convrot_linear_bwd_x_r2(dY, Wq, sw, b, dX, ws)  # noqa: E731
        work = 2.0 * a.M * a.N * a.K
        unit = "TOPS"
    elif a.case == "fwd_lora":
        # forward with an unmerged rank-16 adapter as a bypass in the GEMM epilogue
        x = sg.activations_bf16(0, a.M, a.K, 41, 30.0, dev)
        W = sg.normal_bf16(0, synth.STREAM_W, a.N, a.K, 0.02, dev)
        Wq, sw = cr.convrot_quantize_weight(W, b)
        A, B = sg.lora_pair(0, a.N, a.K, 16, 0.01, dev)
        y = torch.empty((a.M, a.N), dtype=torch.bfloat16, device=dev)
        ws = torch.empty(cr.convrot_linear_lora_workspace_bytes(a.M, a.K, a.N), dtype=torch.uint8, device=dev)
        fn = lambda i: cr.convrot_linear_fwd_lora(x, Wq, sw, b, A, B, 16.0, 1.0, None, y, ws)  # noqa: E731
        work = 2.0 * a.M * a.N * a.K
        unit = "TOPS"
    else:
        T = sg.normal_bf16(0, synth.STREAM_TABLE, a.V, a.D, 0.02, dev)
        Eq, se = cr.convrot_quantize_weight(T, b)
        del T
        ids = [sg.token_ids(0, a.n, a.V, dev, set_index=s) for s in range(8)]
        out = torch.empty((a.n, a.D), dtype=torch.bfloat16, device=dev)
        fn = lambda i: cr.convrot_embedding_lookup(ids[i % 8], Eq, se, b, out)  # noqa: E731
        work = a.n * (8 + a.D + 4 + 2 * a.D)
        unit = "GB/s"

    torch.cuda.synchronize()
    fn(0)
    torch.cuda.synchronize()
    ts = []
    for i in range(a.reps):
        flush.zero_()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        fn(i + 1)
        e1.record()
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1))
    assert cr.convrot_get_error() == cr.OK
    ms = statistics.median(ts)
    rate = work / (ms * 1e-3) / (1e12 if unit == "TOPS" else 1e9)
    print(f"{a.case}: {ms:.4f} ms  {rate:.1f} {unit}")


if __name__ == "__main__":
    main()
