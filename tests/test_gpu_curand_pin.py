"""Pin of the noise words' fourth counter word (the tensor id) against an
independent implementation: cuRAND's device-side Philox4x32-10.

curand_init(seed, subsequence, offset) keys the generator with the 64-bit
seed and positions its 128-bit counter at (offset / 4 as a 64-bit value in
words 0-1, subsequence as a 64-bit value in words 2-3); curand4() returns the
bijection at that counter.  So the noise words of group g at step s and tensor
id t equal curand4 after curand_init(seed, s + 2^32 t, 4 g).  The CPU suite
pins words 0-2 against cuRAND's host generator, which cannot reach word 3.
This test compiles a ten-line kernel that calls cuRAND (a library, not this
project's code) and compares both the oracle's and the library's words."""
import ctypes
import os
import shutil
import subprocess

import numpy as np
import pytest
import torch

import oracle as orc
from semi_structured_sparsity_gb300 import binding as mk
from tests._helpers import assert_bits_equal, bits32

pytestmark = pytest.mark.gpu

SRC = r"""
#include <curand_kernel.h>
#include <stdint.h>
__global__ void draw(unsigned long long seed, const unsigned long long* subseq,
                     const unsigned long long* offset, uint4* out, int n) {
  int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  curandStatePhilox4_32_10_t st;
  curand_init(seed, subseq[i], offset[i], &st);
  out[i] = curand4(&st);
}
extern "C" int curand_words(unsigned long long seed, const unsigned long long* subseq,
                            const unsigned long long* offset, void* out, int n) {
  draw<<<(n + 127) / 128, 128>>>(seed, subseq, offset, (uint4*)out, n);
  return (int)cudaDeviceSynchronize();
}
"""


@pytest.fixture(scope="module")
def curand_lib(tmp_path_factory):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    d = tmp_path_factory.mktemp("curand_pin")
    src = d / "pin.cu"
    src.write_text(SRC)
    so = d / "libpin.so"
    subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O2", "-shared",
                    "-Xcompiler", "-fPIC", "-cudart", "shared", "-o", str(so), str(src)],
                   check=True)
    L = ctypes.CDLL(str(so))
    L.curand_words.argtypes = [ctypes.c_ulonglong, ctypes.c_void_p, ctypes.c_void_p,
                               ctypes.c_void_p, ctypes.c_int]
    L.curand_words.restype = ctypes.c_int
    return L


def test_tensor_id_word_matches_curand_device_philox(curand_lib):
    rng = np.random.default_rng(12)
    n = 4096
    seeds = [0, 0xFFFFFFFFFFFFFFFF, 0x0123456789ABCDEF]
    for seed in seeds:
        step = rng.integers(0, 1 << 32, n, dtype=np.uint64)
        tid = rng.integers(0, 1 << 32, n, dtype=np.uint64)
        group = rng.integers(0, 1 << 40, n, dtype=np.uint64)
        sub = torch.from_numpy((step + (tid << np.uint64(32))).view(np.int64)).cuda()
        off = torch.from_numpy((group * np.uint64(4)).view(np.int64)).cuda()
        out = torch.empty((n, 4), dtype=torch.int32, device="cuda")
        assert curand_lib.curand_words(seed, sub.data_ptr(), off.data_ptr(), out.data_ptr(),
                                       n) == 0
        got = bits32(out)
        want = np.stack([orc.noise_words(seed, int(step[i]), int(tid[i]), int(group[i]), 1)[0]
                         for i in range(n)])
        assert_bits_equal(got, want, "cuRAND vs oracle noise words")
        # and the library's own export at the same coordinates
        for i in range(0, n, 512):
            lib_words = mk.maskllm_noise_words((seed, int(step[i]), int(tid[i])), int(group[i]), 1)
            assert_bits_equal(bits32(lib_words)[0], want[i], "library noise words")
