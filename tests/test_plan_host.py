"""The launch planner (draft_verification_sdv_gb300/csrc/sdv_plan.h) on the
host, without a GPU: a probe built from it with nvcc plans a sweep of shapes,
and the plans must keep the row pass's invariants.  Item mode: chunks cover
the row with no empty chunk, are 128-byte multiples (or the whole row), stay
within 64 per row unless the row needs more 76 KB chunks, and fill at least
four waves of resident warps when the row allows it.  Row mode: exactly when
the rows fill between three quarters and all of one wave of row CTAs (and a
row has a block for each of the CTA's warps), with one chunk per row.  The
select kernel's lanes per row merge: a power of two up to 32, at most the
first power of two at or above the chunks, with every pair and bonus row of a
sequence in one round of its 512 threads."""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))

NSM = 152
ITEM_WARPS = NSM * 4 * 8          # 4 CTAs of 8 warps per SM
ROW_SLOTS = NSM * 8               # 8 row CTAs per SM


def _nvcc():
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    return None


@pytest.fixture(scope="module")
def probe(tmp_path_factory):
    nv = _nvcc()
    if nv is None:
        pytest.skip("nvcc not found")
    exe = str(tmp_path_factory.mktemp("plan") / "plan_probe")
    r = subprocess.run([nv, "-std=c++17", "-O1", os.path.join(HERE, "plan_probe.cu"), "-o", exe],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr

    def run(shapes):
        text = "".join("%d %d %d %d %d %d %d\n" % s for s in shapes)
        out = subprocess.run([exe], input=text, capture_output=True, text=True, check=True).stdout
        return [tuple(int(x) for x in line.split()) for line in out.splitlines()]
    return run


def _shapes():
    out = []
    for V, elt in ((152064, 2), (32000, 2), (5000, 2), (32, 4), (1000, 4), (256, 2)):
        nvec = V * elt // 16
        for B, K, G in ((1, 1, 4), (1, 1, 8), (8, 4, 16), (64, 8, 16), (32, 16, 32), (6, 3, 5),
                        (32, 3, 32), (2, 2, 3), (16, 4, 16), (7, 4, 16)):
            rows = B * K * (2 * G + 1)
            out.append((rows, nvec, ITEM_WARPS, 0, ROW_SLOTS, K, G))
    # row counts around the row-mode window
    for rows in (600, 911, 912, 913, 1056, 1215, 1216, 1217, 2000):
        out.append((rows, 19008, ITEM_WARPS, 0, ROW_SLOTS, 4, 16))
    # a cap on the items (the allocation-free entry point's fixed scratch)
    out.append((4000, 19008, ITEM_WARPS, 40000, ROW_SLOTS, 4, 16))
    return out


def test_plans_keep_the_row_pass_invariants(probe):
    shapes = _shapes()
    for (rows, nvec, warps, max_items, slots, K, G), (chunks, cv, row_mode, lanes) in zip(shapes, probe(shapes)):
        tag = (rows, nvec, max_items)
        want_row = slots * 3 <= 4 * rows <= 4 * slots and nvec >= 4 * 256
        assert row_mode == int(want_row), tag
        if row_mode:
            assert (chunks, cv) == (1, nvec), tag
        else:
            assert cv == nvec or cv % 8 == 0, tag
            assert chunks * cv >= nvec and (chunks - 1) * cv < nvec, tag      # no empty chunk
            assert chunks <= max(64, -(-nvec // 4752)), tag
            if max_items:
                assert rows * chunks <= max(max_items, rows), tag
            else:
                # chunks no larger than four waves of warps ask for (at most
                # 64 chunks a row, at least 64 vectors a chunk), rounded up to
                # a 128-byte multiple
                want = min(64, -(-4 * warps // rows), max(1, nvec // 64))
                want = max(want, -(-nvec // 4752))
                assert cv <= -(-(-(-nvec // want)) // 8) * 8 or cv == nvec, tag
        assert lanes in (1, 2, 4, 8, 16, 32) and (lanes == 1 or lanes // 2 < chunks), tag
        assert (K * G + K) * lanes <= 512 or lanes == 1, tag


def test_self_selection_shape_is_row_mode_and_large_batches_are_not(probe):
    nvec = 152064 * 2 // 16
    res = probe([(8 * 4 * 33, nvec, ITEM_WARPS, 0, ROW_SLOTS, 4, 16),
                 (32 * 16 * 65, nvec, ITEM_WARPS, 0, ROW_SLOTS, 16, 32),
                 (17, nvec, ITEM_WARPS, 0, ROW_SLOTS, 1, 8)])
    assert res[0][:3] == (1, nvec, 1)
    assert res[1][2] == 0 and res[1][0] == 4          # 33 280 rows: four 76 KB chunks
    # 17 rows: split to the cap of 64, whose 297-vector chunks round up to
    # 304 vectors: 63 chunks
    assert res[2][2] == 0 and res[2][:2] == (63, 304)
