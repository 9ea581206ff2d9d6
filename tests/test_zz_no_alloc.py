"""The permutation search entry point that allocates nothing.

maskllm_perm_search_static serves callers that cannot allocate device memory
when they run the search (a runtime that has reserved all device memory for
its own pool, or a host program without a device allocator of its own): its
scratch is a fixed array the library keeps in device memory.  Its results
must be those of maskllm_perm_search with a caller workspace, call after
call, although every call reuses the same array.  This file is collected
last so that a run stopping at the first failure has run every other test.
"""

import os
import subprocess
import sys

import numpy as np
import pytest
import torch

from semi_structured_sparsity_gb300 import binding as mk
from semi_structured_sparsity_gb300 import workloads as W

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    mk.lib()


def _search_c(static, Wt, perm, max_swaps):
    """One search through the C ABI; buffers from torch, pointers to C."""
    L = mk.lib()
    rows, cols = Wt.shape
    swaps = torch.full((max_swaps, 2), -7, dtype=torch.int32, device="cuda")
    gains = torch.full((max_swaps,), -7, dtype=torch.int64, device="cuda")
    small = torch.full((8,), -7, dtype=torch.int32, device="cuda")   # n_swaps, shift
    s = torch.cuda.current_stream().cuda_stream
    if static:
        st = L.maskllm_perm_search_static(Wt.data_ptr(), rows, cols, perm.data_ptr(), max_swaps,
                                          swaps.data_ptr(), gains.data_ptr(), small.data_ptr(),
                                          small.data_ptr() + 16, s)
    else:
        ws = torch.empty((mk.maskllm_perm_workspace_bytes(rows, cols),), dtype=torch.uint8,
                         device="cuda")
        st = L.maskllm_perm_search(Wt.data_ptr(), rows, cols, perm.data_ptr(), max_swaps,
                                   ws.data_ptr(), ws.numel(), swaps.data_ptr(), gains.data_ptr(),
                                   small.data_ptr(), small.data_ptr() + 16, s)
    assert st == 0, mk.maskllm_status_string(st)
    torch.cuda.synchronize()
    n = int(small[0].item())
    return n, swaps[:max(n, 0)].cpu().numpy(), gains[:max(n, 0)].cpu().numpy(), \
        int(small[4].item()), perm.cpu().numpy()


def _case(rows, cols, seed):
    Wt = W.normal_bf16(rows, cols, 0.02, seed, device="cuda")
    g = torch.Generator().manual_seed(seed)
    perm = torch.randperm(cols, generator=g).to(torch.int32).cuda()
    return Wt, perm


# two calls in a row with different shapes (the larger first, so the second
# call runs over what the first left in the shared array), then a third
CASES = [(2048, 1024, 11, 60), (96, 256, 12, 200), (1000, 2048, 13, 20)]


def test_static_scratch_search_matches_workspace_search():
    for rows, cols, seed, max_swaps in CASES:
        Wt, p = _case(rows, cols, seed)
        want = _search_c(False, Wt, p.clone(), max_swaps)
        got = _search_c(True, Wt, p.clone(), max_swaps)
        assert got[0] == want[0] > 0
        for g, w in zip(got[1:], want[1:]):
            assert np.array_equal(g, w)


def test_static_scratch_rejects_shapes_beyond_its_size():
    L = mk.lib()
    Wt, p = _case(3584, 1024, 14)    # needs 32 MiB + 8 KiB of scratch
    small = torch.zeros((8,), dtype=torch.int32, device="cuda")
    st = L.maskllm_perm_search_static(Wt.data_ptr(), 3584, 1024, p.data_ptr(), 5, None, None,
                                      small.data_ptr(), None, torch.cuda.current_stream().cuda_stream)
    assert st == 2    # MASKLLM_ERR_SHAPE
    assert mk.maskllm_perm_workspace_bytes(3584, 1024) > mk.PERM_SEARCH_STATIC_BYTES
    assert mk.maskllm_perm_workspace_bytes(3583, 1024) <= mk.PERM_SEARCH_STATIC_BYTES


def test_static_scratch_call_allocates_no_device_memory():
    """The property the entry point exists for: with its outputs made
    beforehand, a call leaves the device's free memory as it was (a first
    call has loaded the library's device code)."""
    L = mk.lib()
    Wt, p = _case(512, 1024, 15)
    swaps = torch.zeros((40, 2), dtype=torch.int32, device="cuda")
    gains = torch.zeros((40,), dtype=torch.int64, device="cuda")
    small = torch.zeros((8,), dtype=torch.int32, device="cuda")
    s = torch.cuda.current_stream().cuda_stream

    def call(perm):
        st = L.maskllm_perm_search_static(Wt.data_ptr(), 512, 1024, perm.data_ptr(), 40,
                                          swaps.data_ptr(), gains.data_ptr(), small.data_ptr(),
                                          small.data_ptr() + 16, s)
        assert st == 0, mk.maskllm_status_string(st)
        torch.cuda.synchronize()

    first, second = p.clone(), p.clone()
    call(first)
    free_before = torch.cuda.mem_get_info()[0]
    call(second)
    assert torch.cuda.mem_get_info()[0] == free_before
    assert torch.equal(first, second)


_CAPTURE_SCRIPT = r"""
import sys
sys.path.insert(0, {root!r})
import torch
from semi_structured_sparsity_gb300 import binding as mk
from semi_structured_sparsity_gb300 import workloads as W
L = mk.lib()
Wt = W.normal_bf16(64, 256, 0.02, 16, device="cuda")
perm = torch.arange(256, dtype=torch.int32, device="cuda")
small = torch.zeros((8,), dtype=torch.int32, device="cuda")
side = torch.cuda.Stream()
graph = torch.cuda.CUDAGraph()
with torch.cuda.graph(graph, stream=side):
    st = L.maskllm_perm_search_static(Wt.data_ptr(), 64, 256, perm.data_ptr(), 4, None, None,
                                      small.data_ptr(), None, side.cuda_stream)
print("status", st)
st2 = L.maskllm_perm_search_static(Wt.data_ptr(), 64, 256, perm.data_ptr(), 4, None, None,
                                   small.data_ptr(), None, torch.cuda.current_stream().cuda_stream)
torch.cuda.synchronize()
print("after", st2)
"""


def test_static_scratch_first_call_inside_a_capture_is_refused():
    """In a fresh process, a first call made while its stream is being
    captured returns MASKLLM_ERR_INVALID_ARG without launching; the next call
    outside the capture works."""
    r = subprocess.run([sys.executable, "-c", _CAPTURE_SCRIPT.format(root=ROOT)],
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-3000:]
    assert "status 1" in r.stdout and "after 0" in r.stdout, r.stdout
