"""The oracle's Philox4x32-10 stream equals cuRAND's Philox4_32_10 device
generator (a library routine) for the (j, b, 0, 0) counter keying:
curand_init(seed, 0, 4 * (j + 2^32 b)) yields the block of counter (j, b, 0, 0)
under key (seed lo, seed hi)."""
import os
import shutil
import subprocess
import tempfile

import pytest

pytestmark = pytest.mark.gpu

SRC = r"""
#include <cstdio>
#include <curand_kernel.h>
__global__ void draw(unsigned long long seed, unsigned long long offset, uint4* out) {
    curandStatePhilox4_32_10_t st;
    curand_init(seed, 0ull, offset, &st);
    *out = curand4(&st);
}
int main(int argc, char** argv) {
    uint4* d;
    if (cudaMalloc(&d, sizeof(uint4)) != cudaSuccess) return 2;
    unsigned long long seed, j, b;
    while (scanf("%llx %llu %llu", &seed, &j, &b) == 3) {
        draw<<<1, 1>>>(seed, 4ull * (j + (b << 32)), d);
        uint4 h;
        if (cudaMemcpy(&h, d, sizeof h, cudaMemcpyDeviceToHost) != cudaSuccess) return 3;
        printf("%08x %08x %08x %08x\n", h.x, h.y, h.z, h.w);
    }
    return 0;
}
"""


def test_oracle_philox_matches_curand(oracle_lib):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    cases = [(0, 0, 0), (0x0123456789ABCDEF, 3, 7), (42, 31, 0), (2 ** 64 - 1, 5, 63),
             (0xDEADBEEF, 16, 12345), (7, 0, 2 ** 29)]   # offset 4(j + 2^32 b) must fit 64 bits
    with tempfile.TemporaryDirectory() as tmp:
        src, exe = os.path.join(tmp, "p.cu"), os.path.join(tmp, "p")
        with open(src, "w") as f:
            f.write(SRC)
        subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-o", exe, src],
                       check=True, capture_output=True)
        stdin = "".join("%x %d %d\n" % c for c in cases)
        r = subprocess.run([exe], input=stdin, capture_output=True, text=True, check=True)
    lines = r.stdout.strip().splitlines()
    assert len(lines) == len(cases)
    for (seed, j, b), line in zip(cases, lines):
        want = [int(x, 16) for x in line.split()]
        assert oracle_lib.philox4x32_10([j, b, 0, 0], [seed & 0xFFFFFFFF, seed >> 32]) == want
