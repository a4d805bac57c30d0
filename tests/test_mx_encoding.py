"""Bit layouts of the block-scaled MMA's descriptors, checked on the host
before anything runs on a GPU.

The instruction descriptor of tcgen05.mma .kind::mxf8f6f4 / .kind::mxf4 /
.kind::mxf4nvf4 and the shared-memory descriptor that tcgen05.cp reads are
not printed on the pages; the library writes them from the public PTX ISA's
field tables.  This test assembles the expected words field by field from
those tables (name, bit range, value) and compares them with what the
library's encoders return, compiled for the host by nvcc.
"""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "dense_gemm_blackwell_gb300", "csrc")

# (field, first bit, width) of the block-scaled instruction descriptor
IDESC_FIELDS = {"b_sf_id": (4, 2), "a_format": (7, 3), "b_format": (10, 3), "a_major": (15, 1),
                "b_major": (16, 1), "n_dim": (17, 6), "scale_format": (23, 1), "m_dim": (24, 5),
                "a_sf_id": (29, 2)}
# shared-memory matrix descriptor
SDESC_FIELDS = {"start": (0, 14), "lbo": (16, 14), "sbo": (32, 14), "version": (46, 2), "swizzle": (61, 3)}


def assemble(fields, values):
    word = 0
    for name, v in values.items():
        lo, width = fields[name]
        assert 0 <= v < (1 << width), (name, v)
        word |= v << lo
    return word


def nvcc():
    for c in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if c and os.path.exists(c):
            return c
    return None


@pytest.fixture(scope="module")
def encoded(tmp_path_factory):
    cc = nvcc()
    if cc is None:
        pytest.skip("nvcc not available")
    d = tmp_path_factory.mktemp("mxenc")
    src = d / "enc.cu"
    src.write_text(r'''
#include <cstdio>
#include "mx_ptx.cuh"
using namespace dgb;
int main() {
    // (a_format, b_format, M, N, scale_ue8m0, a_mn_major, b_mn_major)
    const unsigned cases[][7] = {{0, 0, 128, 256, 1, 0, 0}, {1, 0, 256, 256, 1, 0, 0}, {0, 1, 128, 128, 1, 0, 0},
                                 {1, 1, 256, 256, 1, 0, 0}, {1, 1, 128, 256, 0, 0, 0}, {1, 1, 256, 256, 0, 0, 0},
                                 {0, 0, 256, 256, 1, 1, 0}, {0, 1, 128, 256, 1, 0, 1}, {1, 0, 256, 256, 1, 1, 1}};
    for (auto& c : cases) {
        unsigned base = make_idesc_block_scaled(c[0], c[1], c[2], c[3], c[4], c[5], c[6]);
        for (unsigned id = 0; id < 4; ++id) printf("I %u %u %u %u %u %u %u %u %u\n", c[0], c[1], c[2], c[3], c[4],
                                                    c[5], c[6], id, idesc_with_scale_ids(base, id));
    }
    const unsigned addrs[] = {0u, 1024u, 0x1F400u, 0x3FFF0u};
    for (unsigned a : addrs) printf("S %u %llu\n", a, (unsigned long long)smem_desc_scale_slab(a));
    return 0;
}
''')
    exe = d / "enc"
    subprocess.run([cc, "-std=c++17", "-I" + CSRC, "-I" + os.path.join(ROOT, "include"), str(src), "-o", str(exe)],
                   check=True, capture_output=True)
    return subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split("\n")


def test_block_scaled_instruction_descriptor(encoded):
    rows = [list(map(int, l.split()[1:])) for l in encoded if l.startswith("I ")]
    assert len(rows) == 36
    for fa, fb, m, n, ue8m0, ma, mb, sf_id, word in rows:
        want = assemble(IDESC_FIELDS, {"a_format": fa, "b_format": fb, "a_major": ma, "b_major": mb,
                                       "n_dim": n >> 3, "scale_format": ue8m0, "m_dim": m >> 4,
                                       "a_sf_id": sf_id, "b_sf_id": sf_id})
        assert word == want, (fa, fb, m, n, ue8m0, sf_id, hex(word), hex(want))
        # sparsity (bit 2), negation (13, 14) and the K-size bit (31, 0 = dense K32 / K64) stay clear
        assert word & ((1 << 2) | (1 << 13) | (1 << 14) | (1 << 31)) == 0


def test_scale_slab_shared_memory_descriptor(encoded):
    rows = [list(map(int, l.split()[1:])) for l in encoded if l.startswith("S ")]
    assert len(rows) == 4
    for addr, word in rows:
        # 32 rows x 16 bytes, no swizzle: 8-row core matrices 128 bytes apart
        want = assemble(SDESC_FIELDS, {"start": (addr >> 4) & 0x3FFF, "lbo": 128 >> 4, "sbo": 128 >> 4,
                                       "version": 1, "swizzle": 0})
        assert word == want, (addr, hex(word), hex(want))
