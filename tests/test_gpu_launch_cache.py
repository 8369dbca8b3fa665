"""The launch-parameter cache (encoded tensor maps and work plans kept per
call signature) must follow the call, not the data: a repeated call with the
same tensors sees their new contents, a call with other tensors of the same
shape uses those tensors, and both keep matching the oracle."""
import pytest
import torch

import oracle
import parity
from transformer_ffn_gb300 import synth

pytestmark = pytest.mark.gpu


def _ffn_oracle(X, inp, act1, act2):
    u = synth.to_u16
    acts = {"relu": oracle.ACT_RELU, "gelu_tanh": oracle.ACT_GELU_TANH, "none": oracle.ACT_NONE}
    return oracle.ffn(u(X), u(inp.W1), u(inp.b1), u(inp.W2), u(inp.b2), acts[act1], acts[act2])


@pytest.mark.parametrize("M,N,O,P", [
    (16, 1024, 2048, 512),      # decode stream
    (100, 512, 1024, 264),      # tensor-core stream
    (300, 256, 1152, 320),      # engine
])
def test_repeated_calls_follow_contents_and_pointers(cuda_lib, M, N, O, P):
    inp = synth.ffn_inputs(M, N, O, P, seed=M + 3, device="cuda")
    Y = torch.empty((M, P), dtype=torch.bfloat16, device="cuda")
    X = inp.X.clone()
    cuda_lib.ffn_forward(X, inp.W1, inp.b1, inp.W2, inp.b2, "gelu_tanh", "none", out=Y)
    cuda_lib.check()
    parity.assert_close(Y.float().cpu().numpy(), _ffn_oracle(X, inp, "gelu_tanh", "none"), "first call")
    # same pointers, new contents: the cached parameters read the new data
    X.copy_(torch.randn_like(X, dtype=torch.float32).to(torch.bfloat16))
    cuda_lib.ffn_forward(X, inp.W1, inp.b1, inp.W2, inp.b2, "gelu_tanh", "none", out=Y)
    cuda_lib.check()
    parity.assert_close(Y.float().cpu().numpy(), _ffn_oracle(X, inp, "gelu_tanh", "none"), "new contents")
    # other tensors of the same shape (other pointers), and another activation
    X2 = inp.X.clone()
    Y2 = torch.empty_like(Y)
    cuda_lib.ffn_forward(X2, inp.W1, inp.b1, inp.W2, inp.b2, "relu", "none", out=Y2)
    cuda_lib.check()
    parity.assert_close(Y2.float().cpu().numpy(), _ffn_oracle(X2, inp, "relu", "none"), "new pointers")
    # many distinct signatures (more than the cache keeps), then the first again
    for i in range(6):
        Xi = inp.X[: max(1, M - i)].clone()
        cuda_lib.ffn_forward(Xi, inp.W1, inp.b1, inp.W2, inp.b2, "gelu_tanh", "none")
    cuda_lib.ffn_forward(X, inp.W1, inp.b1, inp.W2, inp.b2, "gelu_tanh", "none", out=Y)
    cuda_lib.check()
    parity.assert_close(Y.float().cpu().numpy(), _ffn_oracle(X, inp, "gelu_tanh", "none"), "after eviction")


def test_moe_repeated_calls_follow_routing(cuda_lib):
    # the grouped engine's cached parameters are independent of the routing:
    # new logits (another grouping) on the same tensors stay exact
    T, N, O, P, E, k = 300, 128, 384, 192, 8, 2
    inp = synth.moe_inputs(T, N, O, P, E, seed=5, device="cuda")
    u = synth.to_u16
    for router_seed in (1, 2):
        g = torch.Generator(device="cpu").manual_seed(router_seed)
        logits = torch.randn((T, E), generator=g).cuda()
        Y = cuda_lib.moe_ffn_forward(inp.X, logits, k, inp.W1, inp.b1, inp.W2, inp.b2, "gelu_tanh", "none")
        cuda_lib.check()
        want = oracle.moe_ffn(u(inp.X), logits.cpu().numpy(), k, [u(w) for w in inp.W1], [u(b) for b in inp.b1],
                              [u(w) for w in inp.W2], [u(b) for b in inp.b2], oracle.ACT_GELU_TANH, oracle.ACT_NONE)
        parity.assert_close(Y.float().cpu().numpy(), want, f"router seed {router_seed}")
