"""Child process of test_gpu_timeout.py: drives a test build of the library
(short bounded waits, the tile-skip hook) through its C ABI and prints one
JSON line with what it saw.

  python -m tests.timeout_child <path of the test build>

1. a plain varlen call (the reference; checked against the oracle);
2. the same call with one CTA's producer skipping one K/V tile's loads: the
   call must return, and the device error word must hold PA_DEVERR_TIMEOUT;
3. the hook off again: the same call must give the first call's result bit
   for bit, and the error word must be clean.
"""

import ctypes
import json
import sys
import time

import numpy as np
import torch

import oracle
import workloads
from tests.parity import assert_lse_close, assert_out_close

PA_DEVERR_TIMEOUT = 4


class Shape(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in ("num_seqs", "num_q_heads", "num_kv_heads",
                                             "head_size", "block_size", "num_blocks",
                                             "max_blocks_per_seq")]


def main(path):
    L = ctypes.CDLL(path)
    P = ctypes.c_void_p
    L.pa_varlen_fwd.argtypes = [P, P, P, P, P, ctypes.c_int, ctypes.c_int, ctypes.POINTER(Shape),
                                ctypes.c_float, ctypes.c_int, P, P, P]
    L.pa_get_device_error.argtypes = [ctypes.POINTER(ctypes.c_int), P]
    L.pa_test_skip_tile_loads.argtypes = [ctypes.c_int, ctypes.c_int]

    # One request, 768 cached + 256 new tokens, 16 q / 4 kv heads, d 128:
    # 1024 packed rows per kv head, four CTAs; the first CTA of the grid
    # takes the last rows, whose causal context is all 1024 tokens (8 tiles).
    b = workloads.make_paged_batch("timeout", 71, [1024], [256], 16, 4, 128, 16)
    dev = "cuda"
    pool = torch.from_numpy(b.pool.view(np.int16)).to(dev)
    q = torch.from_numpy(b.q.view(np.int16)).to(dev)
    table = torch.from_numpy(b.block_table).to(dev)
    qsl = torch.from_numpy(b.query_start_loc).to(dev)
    seq = torch.from_numpy(b.seq_lens).to(dev)
    shape = Shape(b.num_seqs, b.num_q_heads, b.num_kv_heads, b.head_size, b.block_size,
                  b.num_blocks, b.max_blocks_per_seq)

    def call():
        out = torch.empty_like(q)
        lse = torch.empty((b.num_tokens, b.num_q_heads), dtype=torch.float32, device=dev)
        t0 = time.perf_counter()
        rc = L.pa_varlen_fwd(q.data_ptr(), pool.data_ptr(), table.data_ptr(), qsl.data_ptr(),
                             seq.data_ptr(), b.num_tokens, int(b.query_lens.max()),
                             ctypes.byref(shape), b.scale, 1, out.data_ptr(), lse.data_ptr(),
                             None)
        torch.cuda.synchronize()
        dt = time.perf_counter() - t0
        code = ctypes.c_int(-1)
        rc2 = L.pa_get_device_error(ctypes.byref(code), None)
        return rc, rc2, code.value, out.view(torch.int16).cpu().numpy(), lse.cpu().numpy(), dt

    rec = {}
    rc, rc2, code, out1, lse1, dt = call()
    rec["plain"] = {"status": rc, "err_status": rc2, "device_error": code, "seconds": dt}
    ref_o, ref_l = oracle.paged_attention(b.q, b.pool, b.block_table, b.query_start_loc,
                                          b.seq_lens, b.scale)
    got = workloads.bf16_bits_to_f32(out1.view(np.uint16)).astype(np.float64)
    try:
        rec["plain"]["max_out_err"] = assert_out_close(got, ref_o, "plain call")
        rec["plain"]["max_lse_err"] = assert_lse_close(lse1, ref_l, "plain call lse")
        rec["plain"]["parity"] = True
    except AssertionError as e:
        rec["plain"]["parity"] = str(e)

    assert L.pa_test_skip_tile_loads(0, 1) == 0
    rc, rc2, code, out2, lse2, dt = call()
    assert L.pa_test_skip_tile_loads(-1, -1) == 0
    # Rows of the aborted CTA (q tile 3 of kv head 0: query rows 192-255,
    # q heads 0-3) are invalid; every other row must be untouched.
    keep = np.ones((b.num_tokens, b.num_q_heads), bool)
    keep[192:256, 0:4] = False
    rec["skipped"] = {"status": rc, "err_status": rc2, "device_error": code, "seconds": dt,
                      "other_rows_identical": bool(np.array_equal(out2[keep], out1[keep]) and
                                                   np.array_equal(lse2[keep], lse1[keep])),
                      "aborted_rows_lse_neg_inf": bool(np.isneginf(lse2[~keep]).all())}

    rc, rc2, code, out3, lse3, dt = call()
    rec["after"] = {"status": rc, "err_status": rc2, "device_error": code, "seconds": dt,
                    "bit_identical_to_plain": bool(np.array_equal(out3, out1) and
                                                   np.array_equal(lse3.view(np.uint32),
                                                                  lse1.view(np.uint32)))}
    print(json.dumps(rec), flush=True)


if __name__ == "__main__":
    main(sys.argv[1])
