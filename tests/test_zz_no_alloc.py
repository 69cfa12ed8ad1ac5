"""The entry point that never allocates device memory (attn_fwd_noalloc).

Some callers cannot let a library cudaMalloc: their own memory pool owns all
of device memory from the start (a server that hands the rest of HBM to its
cache), or their path cannot take cudaMalloc's implicit synchronisation of the
device. For them the kernel's one piece of scratch memory, its error word,
lives in a fixed array compiled into the library, and
attn_noalloc_last_device_error reads that word without allocating either.

These tests call the entry point through the C ABI twice in a row (the second
call reuses the array the first one left behind) and check each result against
attn_fwd's single-kernel path (split=False, the same kernel and schedule) bit
for bit; they make one call's wait run out and read ATTN_ERR_TIMEOUT back from
the array; and, in a fresh process that never calls attn_fwd, they check that
a call changes neither the device's free memory nor torch's reserved memory.
The file is collected last so that a stop-at-first-failure run has already run
every other test.
"""
import json
import os
import subprocess
import sys

import pytest
import torch

import exact_long_sequence_gb300 as ela
from exact_long_sequence_gb300 import workloads

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


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
        o_ref, l_ref = ela.attn_fwd(q, k, v, causal=causal, split=False)
        o = torch.full_like(q, float("nan"))
        lse = torch.full(q.shape[:3], float("nan"), dtype=torch.float32, device="cuda")
        ela.attn_fwd_noalloc(q, k, v, o, lse, causal=causal)
        assert ela.noalloc_last_device_error() == ela.ATTN_OK, f"call {call}"
        assert torch.equal(o, o_ref) and torch.equal(lse, l_ref), f"call {call}"


def test_noalloc_reports_a_timeout_through_its_own_reader():
    q, k, v = (t.cuda() for t in workloads.make_inputs(1, 2, 512, 128, seed=23))
    o_ref, l_ref = ela.attn_fwd(q, k, v, split=False)
    o, lse = torch.empty_like(q), torch.empty(q.shape[:3], dtype=torch.float32, device="cuda")
    assert ela.debug_arm_timeout(20_000_000) == ela.ATTN_OK
    ela.attn_fwd_noalloc(q, k, v, o, lse)
    assert ela.noalloc_last_device_error() == ela.ATTN_ERR_TIMEOUT
    assert ela.noalloc_last_device_error() == ela.ATTN_OK  # the reader cleared the word
    ela.attn_fwd_noalloc(q, k, v, o, lse)
    assert ela.noalloc_last_device_error() == ela.ATTN_OK
    assert torch.equal(o, o_ref) and torch.equal(lse, l_ref)


FRESH_PROCESS = r"""
import json, sys
import torch
sys.path.insert(0, ROOT)
import exact_long_sequence_gb300 as ela
from exact_long_sequence_gb300 import workloads

q, k, v = (t.cuda() for t in workloads.make_inputs(1, 4, 2048, 128, seed=24))
o, lse = torch.empty_like(q), torch.empty(q.shape[:3], dtype=torch.float32, device="cuda")
ela.load_library()
# the first call on the device does its one-time set-up (and loads the kernel's module)
ela.attn_fwd_noalloc(q, k, v, o, lse, causal=True)
first = ela.noalloc_last_device_error()
torch.cuda.synchronize()
before = (torch.cuda.mem_get_info()[0], torch.cuda.memory_reserved())
ela.attn_fwd_noalloc(q, k, v, o, lse, causal=True)
second = ela.noalloc_last_device_error()
torch.cuda.synchronize()
after = (torch.cuda.mem_get_info()[0], torch.cuda.memory_reserved())
o_ref, l_ref = ela.attn_fwd(q, k, v, causal=True, split=False)
torch.cuda.synchronize()
print(json.dumps({"first": first, "second": second, "before": before, "after": after,
                  "equal": bool(torch.equal(o, o_ref) and torch.equal(lse, l_ref))}))
""".replace("ROOT", repr(ROOT))


def test_noalloc_allocates_nothing_in_a_fresh_process():
    r = subprocess.run([sys.executable, "-c", FRESH_PROCESS], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    out = json.loads(r.stdout.strip().splitlines()[-1])
    assert out["first"] == ela.ATTN_OK and out["second"] == ela.ATTN_OK, out
    assert out["before"] == out["after"], out
    assert out["equal"], out
