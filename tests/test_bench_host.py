"""CPU checks of bench.py's bookkeeping: the recorded ncu traffic stays tied
to the GEMM kernel it was measured on."""
import os
import sys

from helpers import ROOT

sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _reader(patch=None):
    def read(f):
        data = open(os.path.join(ROOT, f), "rb").read()
        return patch(f, data) if patch else data
    return read


def test_digest_ignores_comments_and_row_kernels():
    base = bench.gemm_source_digest(_reader())

    def comment(f, data):
        return data.replace(b"namespace w4a8 {", b"namespace w4a8 {\n// a note\n/* another */", 1) \
            if f.endswith("moe.cu") else data

    def row_kernel(f, data):
        if not f.endswith("moe.cu"):
            return data
        a = data.index(b"\n", data.index(b"// Gather: ")) + 1   # inside the row-kernel part
        return data[:a] + b"__device__ int unrelated_row_helper;\n" + data[a:]

    assert bench.gemm_source_digest(_reader(comment)) == base
    assert bench.gemm_source_digest(_reader(row_kernel)) == base


def test_digest_changes_with_the_gemm_code():
    base = bench.gemm_source_digest(_reader())

    def gemm(f, data):
        return data.replace(b"constexpr int kClaimRounds = 2;", b"constexpr int kClaimRounds = 3;", 1) \
            if f.endswith("moe.cu") else data

    def header(f, data):
        return data + b"\n#define W4A8_SOMETHING 1\n" if f.endswith("ptx.cuh") else data

    assert bench.gemm_source_digest(_reader(gemm)) != base
    assert bench.gemm_source_digest(_reader(header)) != base


def test_recorded_traffic_matches_the_sources():
    """The committed traffic records belong to the committed GEMM (else the
    bench reports null): each launch moves at least its algorithmic bytes."""
    alg = {"grok_prefill:gate_up": 8 * (65536 * 3072 + 65536 * 4),
           "mixtral_decode:one_launch": 705_691_648}
    assert bench.NCU_TRAFFIC["sha256"] == bench.gemm_source_digest()
    for key, nbytes in alg.items():
        t = bench.ncu_traffic(key)
        assert t is not None and t >= nbytes, key
