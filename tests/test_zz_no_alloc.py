"""GPU check of fa_bwd_noalloc, the backward entry point that allocates
nothing and uses the library's own device workspace instead of one passed
by the caller (for callers that must not allocate at the point of the
call).  It runs the same kernels as fa_bwd, so its gradients must equal
fa_bwd's bit for bit; two calls in a row check that the reused workspace
carries nothing from one call into the next.  The file is named to be
collected last, so it also runs after every other test in one session.
"""
import pytest
import torch

import exact_attention_forward_fa_gb300 as fa
from exact_attention_forward_fa_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("B,H,N,d,causal", [(2, 3, 1000, 128, True), (1, 4, 777, 64, False)])
def test_noalloc_matches_fa_bwd_twice(gpu_lib, B, H, N, d, causal):
    dev = torch.device("cuda")
    q, k, v = (x.to(dev) for x in synth.qkv(B, H, N, d, seed=N))
    dout = torch.from_numpy(synth.normal((B, N, H, d), seed=N + 3)).to(q.dtype).to(dev)
    a = synth.default_alpha(d)
    o, lse = gpu_lib.attention(q, k, v, causal=causal, alpha=a)
    ref = gpu_lib.attention_backward(q, k, v, o, lse, dout, causal=causal, alpha=a)
    for _ in range(2):
        g = [torch.full_like(q, float("nan")) for _ in range(3)]
        rc = gpu_lib.fa_bwd_noalloc(q, k, v, o, dout, lse, *g, B, H, N, d, a, int(causal),
                                    gpu_lib.FA_BF16)
        assert rc == gpu_lib.FA_OK
        assert gpu_lib.fa_check_status() == gpu_lib.FA_OK
        for x, y in zip(g, ref):
            assert torch.equal(x, y)
