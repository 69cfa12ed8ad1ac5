"""The entry point that never allocates device memory (attn_fwd_noalloc).

Some callers cannot let a library cudaMalloc: their own pool owns all of device
memory, or their path cannot take cudaMalloc's implicit synchronisation. For
them the kernel's one piece of scratch memory, its error word, lives in a fixed
array compiled into the library. This test calls that entry point through the
C ABI twice in a row (the second call reuses the array the first one left
behind) and checks each result against attn_fwd's, within the parity
tolerances. It is collected last so that a stop-at-first-failure run has
already run every other test.
"""
import pytest
import torch

import exact_long_sequence_gb300 as ela
from exact_long_sequence_gb300 import workloads

pytestmark = pytest.mark.gpu

O_TOL = 2e-2
LSE_RTOL = 1e-3


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from exact_long_sequence_gb300 import _build

    _build.build()
    ela.load_library()


@pytest.mark.parametrize("causal,d", [(False, 128), (True, 64)])
def test_noalloc_matches_attn_fwd_on_two_calls_in_a_row(causal, d):
    for call, (N, seed) in enumerate([(1000, 21), (300, 22)]):
        q, k, v = (t.cuda() for t in workloads.make_inputs(2, 3, N, d, seed=seed))
        o_ref, l_ref = ela.attn_fwd(q, k, v, causal=causal)
        o = torch.full_like(q, float("nan"))
        lse = torch.full(q.shape[:3], float("nan"), dtype=torch.float32, device="cuda")
        ela.attn_fwd_noalloc(q, k, v, o, lse, causal=causal)
        torch.cuda.synchronize()
        assert not torch.isnan(o).any() and not torch.isnan(lse).any(), f"call {call}: unwritten output"
        assert (o.float() - o_ref.float()).abs().max().item() <= O_TOL, f"call {call}"
        assert ((lse - l_ref).abs() / l_ref.abs()).max().item() <= LSE_RTOL, f"call {call}"
