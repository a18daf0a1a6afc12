"""The bounded-wait failure path of the tensor-core kernels, made to run out.

Every mbarrier wait of the tcgen05 kernels polls a bounded number of times;
on timeout the thread records PA_DEVERR_TIMEOUT, raises the CTA's abort
flag, and every role leaves its loop, waits (bounded) for its own copies and
MMAs in flight, frees its TMEM and returns.  A correct kernel never gets
there, so the test builds a variant of the library (not the default build)
with a short poll limit and a hook under which the TMA producer of one CTA
of the varlen kernel issues neither the copies nor the byte count of one
K/V tile: that tile's barriers are then a flag that nothing sets, and the
waits on them can only end at their limit.  Nothing is left in flight --
the copies that were issued land before the producer leaves, and the MMA
thread waits for its own MMAs -- so the kernel returns and the context stays
usable.

The variant runs in a child process (tests/timeout_child.py); the test
checks that the call returned, that the error word says PA_DEVERR_TIMEOUT,
that the other CTAs' rows are untouched, and that the next normal call gives
the same bits as the call before the failure.
"""

import json
import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def test_lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_50_gb300 import build
    return build.build(extra_flags=["-DPA_TEST_HOOKS", "-DPA_WAIT_POLLS=4096"],
                       out_dir=os.path.join(build.PKG, "_build", "timeout_variant"),
                       lib_name="libpa_timeout.so")


def test_skipped_tile_times_out_and_the_device_recovers(test_lib):
    r = subprocess.run([sys.executable, "-m", "tests.timeout_child", test_lib], cwd=ROOT,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    rec = json.loads(r.stdout.strip().splitlines()[-1])
    plain, skipped, after = rec["plain"], rec["skipped"], rec["after"]
    assert plain["status"] == 0 and plain["err_status"] == 0 and plain["device_error"] == 0
    assert plain["parity"] is True, plain          # the plain call matches the oracle
    # The launch itself succeeds; the device error word reports the timeout.
    assert skipped["status"] == 0 and skipped["err_status"] == 0, skipped
    assert skipped["device_error"] & 4, skipped
    assert skipped["other_rows_identical"] and skipped["aborted_rows_lse_neg_inf"], skipped
    # The context is still usable and nothing stale is left behind.
    assert after["status"] == 0 and after["device_error"] == 0, after
    assert after["bit_identical_to_plain"], after
