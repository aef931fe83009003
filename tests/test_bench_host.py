"""Host-side pieces of bench.py: the oracle sample both CPU timings share, and the
reference arm's JSON line (it runs the oracle only, so it needs no GPU)."""
import json
import math

import pytest


@pytest.mark.parametrize("cores", [1, 2, 3, 4, 6, 8, 12, 16, 24, 64, 72])
@pytest.mark.parametrize("nh,B", [(1, 5), (3, 32), (6, 32), (6, 128), (3, 4)])
def test_oracle_sample_fills_cores(cores, nh, B):
    import bench
    from visual_backbone_gb300 import synth
    wl = synth.Workload("w", B, 4, 4, nh, 16, 0, "f32")
    n = bench.oracle_images(wl, cores)
    assert 1 <= n <= B
    if n < B:
        # every core gets the same number of (image, head) jobs, and no fewer images do
        assert (n * nh) % cores == 0
        assert all((m * nh) % cores for m in range(1, n))
    else:
        assert n == min(B, math.lcm(cores, nh) // nh)


def test_reference_arm_line(orc, capsys):
    import bench
    rc = bench.main(["--impl", "reference", "--workload", "tiny", "--steps", "2", "--warmup", "3"])
    assert rc in (0, None)
    lines = [l for l in capsys.readouterr().out.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["steps"] == 2 and d["warmup"] == 3
    assert d["value"] > 0 and d["higher_is_better"] is True
    assert d["cpu_baseline"]["value"] == d["value"] and d["cpu_baseline"]["kind"] == "oracle"
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
