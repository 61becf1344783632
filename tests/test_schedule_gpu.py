"""w4g128_schedule over a spread of calls: what it reports agrees with the
workspace query and with the schedule rules the kernels rely on, and every
call it describes runs and matches the oracle's bound."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import int4_weight_only_g128_gb300 as w  # noqa: E402
import synth  # noqa: E402
from gpu_helpers import SEED, DevMatrix, check_against_oracle, run  # noqa: E402

LAYER = [(5120, 6144)] * 3 + [(6144, 5120), (5120, 34816), (17408, 5120)]
SINGLE = [(128, 16), (640, 80), (4096, 4096), (5120, 6144), (17408, 5120), (8192, 4096), (65536, 208),
          (5120, 248320)]


def segs_quads(K, N):
    return -(-K // 512), -(-N // 64)


@pytest.mark.gpu
@pytest.mark.parametrize("M", [1, 2, 8, 9, 16])
@pytest.mark.parametrize("shapes", [[s] for s in SINGLE] + [LAYER, [(128, 16), (640, 80), (4096, 4096)]],
                         ids=lambda s: "+".join(f"{k}x{n}" for k, n in s))
def test_schedule_invariants(shapes, M):
    descs = [(None, None, None, K, N) for K, N in shapes]
    s = w.w4g128_schedule(descs, M)
    items = sum(a * b for a, b in (segs_quads(K, N) for K, N in shapes))
    assert s["items"] == items
    assert s["workspace_bytes"] == w.w4g128_decode_step_workspace_bytes(descs, M) > 0
    if len(shapes) == 1:
        K, N = shapes[0]
        assert s["workspace_bytes"] == w.w4g128_workspace_bytes(M, K, N)
    assert s["ctas"] >= 1 and 1 <= s["cta_warps"] <= (8 if M > 8 else 16)
    assert s["ring_depth"] >= 2
    if M == 1:
        assert s["second_pass"] in (0, 1)
    else:
        assert s["local"] == 0 and s["pair_quads"] == 0 and s["second_pass"] in (2, 3)
    if s["pair_quads"]:
        assert len(shapes) == 1 and s["local"] == 1 and s["second_pass"] == 0
        S, NQ = segs_quads(*shapes[0])
        assert s["ctas"] == 2 * NQ and s["cta_warps"] == -(-S // 2)
    if not s["local"]:
        # the balanced split: every streaming warp has at least one item
        assert (s["ctas"] - 1) * s["cta_warps"] < items


@pytest.mark.gpu
@pytest.mark.parametrize("K,N", [(4096, 4096), (8192, 4096), (640, 80)])
def test_described_call_runs(K, N):
    """The call a schedule describes runs: within the oracle's bound, status clear."""
    mat = DevMatrix(K, N, matrix_id=3200 + K // 128)
    x = synth.x(SEED, 3201 + K, 1, K)
    assert w.w4g128_schedule([(mat.packed, None, None, K, N)], 1)["local"] == 1
    check_against_oracle(run(mat, x), x, mat.codes, mat.scales, mat.mins)
