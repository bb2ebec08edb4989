"""The layer's calls inside a captured CUDA graph.

Every entry point only enqueues work on the caller's stream (no allocation, no
synchronisation), so a training step of the layer can be captured once and
replayed; the replay must give exactly the bits of the eager calls."""
import pytest

import synth
from helpers import torch_bf16

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import int8_rotated_quantized_gb300 as cr  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    cr._build.build()
    cr.lib()


def test_step_replays_from_a_cuda_graph():
    M, K, N, b = 300, 512, 384, 128
    x = torch_bf16(synth.activations_bf16(31, M, K, 4, 20.0))
    W = torch_bf16(synth.normal_bf16(31, synth.STREAM_W, N, K, 0.02))
    dY = torch_bf16(synth.normal_bf16(31, synth.STREAM_DY, M, N, 1e-3))
    Wq, sw = cr.convrot_quantize_weight(W, b)
    WtQ, swt = cr.convrot_prepare_bwd_weight(Wq, sw, b)
    ws = torch.empty(max(cr.convrot_linear_workspace_bytes(M, K, N), cr.convrot_linear_workspace_bytes(M, N, K)),
                     dtype=torch.uint8, device="cuda")
    y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    dX = torch.empty((M, K), dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):  # eager calls first: per-device launch parameters are cached before capture
        cr.convrot_linear_fwd(x, Wq, sw, b, y=y, workspace=ws, stream=s)
        cr.convrot_linear_bwd_x(dY, WtQ, swt, b, dX=dX, workspace=ws, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    y_eager, dx_eager = y.clone(), dX.clone()
    y.zero_()
    dX.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        st = torch.cuda.current_stream()
        cr.convrot_linear_fwd(x, Wq, sw, b, y=y, workspace=ws, stream=st)
        cr.convrot_linear_bwd_x(dY, WtQ, swt, b, dX=dX, workspace=ws, stream=st)
    for _ in range(2):
        y.zero_()
        dX.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(y, y_eager) and torch.equal(dX, dx_eager)
    assert cr.convrot_get_error() == cr.OK


def test_lora_bypass_forward_replays_from_a_cuda_graph():
    """The forward with an unmerged adapter launches four kernels (activation quantizer, bypass operands,
    weight widening, GEMM) on the caller's stream with a caller workspace: capturable, and the replay gives the
    eager bits."""
    M, K, N, b, r = 300, 1024, 272, 128, 16
    x = torch_bf16(synth.activations_bf16(37, M, K, 4, 20.0))
    W = torch_bf16(synth.normal_bf16(37, synth.STREAM_W, N, K, 0.02))
    A, B = synth.lora_pair(37, N, K, r, 0.05)
    A, B = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    bias = torch_bf16(synth.normal_bf16(37, 9, 1, N, 0.5)[0])
    Wq, sw = cr.convrot_quantize_weight(W, b)
    ws = torch.empty(cr.convrot_linear_lora_workspace_bytes(M, K, N), dtype=torch.uint8, device="cuda")
    y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):  # eager call first: launch parameters are cached before capture
        cr.convrot_linear_fwd_lora(x, Wq, sw, b, A, B, 16.0, 1.0, bias=bias, y=y, workspace=ws, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    y_eager = y.clone()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        cr.convrot_linear_fwd_lora(x, Wq, sw, b, A, B, 16.0, 1.0, bias=bias, y=y, workspace=ws,
                                   stream=torch.cuda.current_stream())
    for _ in range(2):
        y.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(y, y_eager)
    assert cr.convrot_get_error() == cr.OK


def test_bf16_and_second_reading_backward_replay_from_a_cuda_graph():
    """The two other backward calls (the bf16 mode: transient weight + bf16 GEMM; the second reading of the int8
    backward: four kernels) with caller workspaces: capturable, and the replays give the eager bits."""
    M, N, K, b = 150, 512, 384, 128
    W = torch_bf16(synth.normal_bf16(41, synth.STREAM_W, N, K, 0.02))
    dY = torch_bf16(synth.normal_bf16(41, synth.STREAM_DY, M, N, 1e-3))
    Wq, sw = cr.convrot_quantize_weight(W, b)
    ws1 = torch.empty(cr.convrot_bwd_x_bf16_workspace_bytes(N, K), dtype=torch.uint8, device="cuda")
    ws2 = torch.empty(cr.convrot_bwd_x_r2_workspace_bytes(M, N, K), dtype=torch.uint8, device="cuda")
    d1 = torch.empty((M, K), dtype=torch.bfloat16, device="cuda")
    d2 = torch.empty((M, K), dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        cr.convrot_linear_bwd_x_bf16(dY, Wq, sw, b, dX=d1, workspace=ws1, stream=s)
        cr.convrot_linear_bwd_x_r2(dY, Wq, sw, b, dX=d2, workspace=ws2, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    e1, e2 = d1.clone(), d2.clone()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        st = torch.cuda.current_stream()
        cr.convrot_linear_bwd_x_bf16(dY, Wq, sw, b, dX=d1, workspace=ws1, stream=st)
        cr.convrot_linear_bwd_x_r2(dY, Wq, sw, b, dX=d2, workspace=ws2, stream=st)
    for _ in range(2):
        d1.zero_()
        d2.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(d1, e1) and torch.equal(d2, e2)
    assert cr.convrot_get_error() == cr.OK
