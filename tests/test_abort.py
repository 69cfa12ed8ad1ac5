"""The forward kernel's own abort path, driven on the GPU without a fault.

Every wait in the kernel is bounded.  attn_debug_arm_timeout arms a one-shot
for the next forward launch: a short wait limit, and CTA 0 arms the barrier of
its first query-tile copy without issuing the copy.  The MMA warp's wait on
that barrier runs out; it records ATTN_ERR_TIMEOUT and raises the CTA's abort
flag, the producer and the softmax warpgroups leave their loops at their next
wait, the producer waits (bounded) for its copies in flight, the MMA warp
waits for its MMAs, and tensor memory is freed before the kernel returns.

Each case checks that the status comes back as ATTN_ERR_TIMEOUT, that the
launch ended well before the default 4 s limit, and that the context is still
usable: the next launch, unarmed, reproduces the result of a launch made
before the abort bit for bit (every path here is deterministic) and reports
ATTN_OK.  The single-CTA case is also compared with the fp64 oracle.
"""
import time

import numpy as np
import pytest
import torch

import exact_long_sequence_gb300 as ela
from exact_long_sequence_gb300 import workloads

pytestmark = pytest.mark.gpu

LIMIT_NS = 20_000_000  # 20 ms


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from exact_long_sequence_gb300 import _build

    _build.build()
    ela.load_library()


CASES = [  # B, H, N, d, causal, split, what it exercises
    (1, 1, 256, 128, False, False, "one CTA, static schedule"),
    (1, 4, 4096, 64, False, False, "64 CTAs, static schedule, the K/V ring full when the abort comes"),
    (1, 8, 8192, 128, True, True, "causal, 256 units on the dynamic schedule (item ring)"),
    (1, 1, 1000, 64, False, True, "K/V split: segments and their in-kernel merge"),
]


@pytest.mark.parametrize("B,H,N,d,causal,split,what", CASES)
def test_abort_reports_timeout_and_the_next_launch_is_unchanged(B, H, N, d, causal, split, what):
    q, k, v = (t.cuda() for t in workloads.make_inputs(B, H, N, d, seed=40 + N))
    o_ref, l_ref = ela.attn_fwd(q, k, v, causal=causal, split=split)
    assert ela.last_device_error() == ela.ATTN_OK
    o_ref, l_ref = o_ref.clone(), l_ref.clone()

    assert ela.debug_arm_timeout(LIMIT_NS) == ela.ATTN_OK
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    ela.attn_fwd(q, k, v, causal=causal, split=split)
    status = ela.last_device_error()
    elapsed = time.perf_counter() - t0
    assert status == ela.ATTN_ERR_TIMEOUT, f"{what}: status {status}"
    assert elapsed < 1.5, f"{what}: the aborted launch took {elapsed:.2f} s"

    o, lse = ela.attn_fwd(q, k, v, causal=causal, split=split)
    assert ela.last_device_error() == ela.ATTN_OK, what
    assert torch.equal(o, o_ref) and torch.equal(lse, l_ref), what


def test_abort_then_oracle_parity(oracle_mod):
    q, k, v = workloads.make_inputs(1, 2, 300, 128, seed=77)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    assert ela.debug_arm_timeout(LIMIT_NS) == ela.ATTN_OK
    ela.attn_fwd(qd, kd, vd, causal=True, split=False)
    assert ela.last_device_error() == ela.ATTN_ERR_TIMEOUT
    o, lse = ela.attn_fwd(qd, kd, vd, causal=True, split=False)
    assert ela.last_device_error() == ela.ATTN_OK
    O, L = oracle_mod.attention_rows(q, k, v, True, ela.default_scale(128))
    assert np.abs(o.double().cpu().numpy().reshape(O.shape) - O).max() <= 2e-2
    assert (np.abs(lse.double().cpu().numpy().reshape(L.shape) - L) <= 1e-3 * np.abs(L)).all()
