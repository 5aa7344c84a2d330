"""fa_naive_fwd_noalloc: the standard-attention path for callers that cannot
allocate device memory (needs a GB300).

The entry point keeps its N x N matrices in a fixed 64 MiB array inside the
library instead of a caller-provided workspace, for services that reserve all
device memory up front or code paths where an allocation is not allowed. Its
results must equal those of fa_naive_fwd, which takes a workspace, on two
calls in a row (the array is shared and keeps the previous call's contents).
This file is collected last on purpose.
"""
import ctypes
import gc
import math

import pytest
import torch

from exact_io_aware_34_gb300 import fa, inputs

pytestmark = pytest.mark.gpu

LIMIT = 64 << 20


def _noalloc(lib, q, k, v, o, lse, scale, stream=None):
    B, H, N, d = q.shape
    return lib.fa_naive_fwd_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                    B, H, N, d, ctypes.c_float(scale), stream)


@pytest.mark.parametrize("d", [64, 128])
def test_noalloc_matches_workspace_entry_twice(d):
    lib = fa.load_library()
    shapes = [(2, 3, 1000, 7), (1, 4, 777, 8)]          # (B, H, N, seed): two different calls in a row
    for B, H, N, seed in shapes:
        assert fa.fa_naive_workspace_bytes(B, H, N) <= LIMIT
        q, k, v = (x.cuda() for x in inputs.make_random(B, H, N, d, seed=seed + d))
        s = 1 / math.sqrt(d)
        o_ref, lse_ref = fa.fa_naive_fwd(q, k, v, scale=s)            # existing entry point, own workspace
        o = torch.empty_like(q)
        lse = torch.empty(B, H, N, dtype=torch.float32, device="cuda")
        gc.collect()
        torch.cuda.synchronize()
        before = torch.cuda.memory_allocated()
        assert _noalloc(lib, q, k, v, o, lse, s) == fa.FA_OK
        torch.cuda.synchronize()
        assert torch.cuda.memory_allocated() <= before      # nothing was allocated through torch
        assert fa.fa_get_device_status()[0] == fa.FA_OK
        # The same three deterministic kernels on the same inputs, with only
        # the scratch memory moved: the results are equal bit for bit.
        assert torch.equal(o.view(torch.int16), o_ref.view(torch.int16))
        assert torch.equal(lse.view(torch.int32), lse_ref.view(torch.int32))


def test_noalloc_makes_no_device_allocation():
    """After the first call on the device, further calls leave free device memory unchanged."""
    lib = fa.load_library()
    q, k, v = (x.cuda() for x in inputs.make_random(1, 2, 512, 128, seed=11))
    o = torch.empty_like(q)
    lse = torch.empty(1, 2, 512, dtype=torch.float32, device="cuda")
    assert _noalloc(lib, q, k, v, o, lse, 0.08) == fa.FA_OK
    gc.collect()
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        assert _noalloc(lib, q, k, v, o, lse, 0.08) == fa.FA_OK
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0


def test_noalloc_rejects_requests_beyond_the_array():
    lib = fa.load_library()
    N = 8192                                   # one head needs 128 MiB of scores
    assert fa.fa_naive_workspace_bytes(1, 1, N) > LIMIT
    q = torch.zeros(1, 1, N, 64, dtype=torch.bfloat16, device="cuda")
    o = torch.empty_like(q)
    lse = torch.empty(1, 1, N, dtype=torch.float32, device="cuda")
    assert _noalloc(lib, q, q.clone(), q.clone(), o, lse, 0.1) == fa.FA_ERR_UNSUPPORTED
