"""The benchmark's reference arm on the CPU: `bench.py --impl reference` times the oracle and
prints one JSON line with the keys the measurement contract names (no GPU needed)."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_contract_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--steps", "1", "--warmup", "0"],
                         cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference"
    assert d["metric"] == "Groth16 H computations/s at 2^18" and d["unit"] == "H/s"
    assert d["value"] > 0 and d["higher_is_better"] is True
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0


def _bench():
    if ROOT not in sys.path:
        sys.path.insert(0, ROOT)
    import bench

    return bench


def test_per_kernel_work_sums_to_the_whole_h():
    # The roofline's per-launch work, summed over one serialized H's launch census (two
    # gathers, the slice kernels of each level, the join), is the whole H's count, so the
    # whole-step fraction is h_ops / step time / peak and nothing is counted twice.
    bench = _bench()
    for k in (6, 12, 14, 17, 18, 22, 23, 27):
        for from_witness in (True, False):
            nnz_a, nnz_b = (296223, 443023) if from_witness else (0, 0)
            want = bench.h_ops(k, nnz_a, nnz_b, from_witness)
            per_kernel = bench.kernel_ops_per_h(k, nnz_a, nnz_b, from_witness)
            assert sum(per_kernel.values()) == want
            census = bench.launches_per_h(k, from_witness)
            assert set(census) == set(per_kernel)
            got = sum(bench.algorithmic_ops(name, k, nnz_a, nnz_b, from_witness) * count
                      for name, count in census.items())
            assert got == want, (k, from_witness)


def test_h_ops_is_the_multiply_count_of_the_method():
    # The method's count at 2^18: 6 (n/2) k butterflies + 3n (1/n) + 3n (shift) + n (join)
    # + nnz_A + nnz_B + n (gather, c = a * b) multiplies, n reductions.
    bench = _bench()
    n, k, nnz_a, nnz_b = 1 << 18, 18, 296223, 443023
    mm = 6 * (n // 2) * k + 3 * n + 3 * n + n + nnz_a + nnz_b + n
    assert mm == 16992174  # 16.99 M multiplies
    assert bench.h_ops(k, nnz_a, nnz_b) == mm * (2 * 128 + 8) + n * (2 * 64 + 8)
    # each gather launch is charged its own matrix only
    assert bench.algorithmic_ops("gather_a", k, nnz_a, nnz_b) == nnz_a * 264
    assert bench.algorithmic_ops("gather_b", k, nnz_a, nnz_b) == nnz_b * 264
