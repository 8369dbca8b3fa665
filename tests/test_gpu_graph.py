"""The forward calls captured into a CUDA graph and replayed.

Ready flags are compared against an epoch kept on the device and advanced by
every launch, so a replayed launch (whose parameters are frozen at capture)
still waits for this replay's hidden tiles.  Each replay gets new input and
must reproduce the eager call bit for bit (the kernels are deterministic).
"""
import pytest
import torch

from transformer_ffn_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("shape,path", [((300, 256, 1024, 512), 1), ((16, 512, 1024, 256), 2),
                                        ((520, 128, 768, 264), 1), ((100, 512, 2048, 512), 6)])
def test_replayed_ffn_matches_eager(cuda_lib, shape, path):
    tffn = cuda_lib
    M, N, O, P = shape
    inp = synth.ffn_inputs(M, N, O, P, seed=31, device="cuda")
    old = tffn.set_option(tffn.OPT_PATH, path)
    try:
        X = inp.X.clone()
        out = torch.empty((M, P), dtype=torch.bfloat16, device="cuda")
        tffn.ffn_forward(X, inp.W1, inp.b1, inp.W2, inp.b2, "gelu_tanh", "none", out=out)   # warm: workspace
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            tffn.ffn_forward(X, inp.W1, inp.b1, inp.W2, inp.b2, "gelu_tanh", "none", out=out)
        for i in range(4):
            Xi = synth.ffn_inputs(M, N, O, P, seed=100 + i, device="cuda").X
            X.copy_(Xi)
            g.replay()
            torch.cuda.synchronize()
            want = tffn.ffn_forward(Xi, inp.W1, inp.b1, inp.W2, inp.b2, "gelu_tanh", "none")
            tffn.check()
            assert torch.equal(out, want), f"replay {i}"
    finally:
        tffn.set_option(tffn.OPT_PATH, old)


def test_replayed_moe_matches_eager(cuda_lib):
    tffn = cuda_lib
    T, N, O, P, E, k = 200, 128, 512, 256, 8, 2
    inp = synth.moe_inputs(T, N, O, P, E, seed=32, device="cuda")
    X = inp.X.clone()
    L = inp.logits.clone()
    out = torch.empty((T, P), dtype=torch.bfloat16, device="cuda")
    tffn.moe_ffn_forward(X, L, k, inp.W1, inp.b1, inp.W2, inp.b2, out=out)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        tffn.moe_ffn_forward(X, L, k, inp.W1, inp.b1, inp.W2, inp.b2, out=out)
    for i in range(3):
        nxt = synth.moe_inputs(T, N, O, P, E, seed=200 + i, device="cuda")
        X.copy_(nxt.X)
        L.copy_(nxt.logits)
        g.replay()
        torch.cuda.synchronize()
        want = tffn.moe_ffn_forward(nxt.X, nxt.logits, k, inp.W1, inp.b1, inp.W2, inp.b2)
        tffn.check()
        assert torch.equal(out, want), f"replay {i}"
