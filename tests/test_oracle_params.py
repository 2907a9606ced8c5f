"""Pins for the oracle's parameter selection (gMAGNUS Sec. III-D, Eqs. (4)-(7)).

The chunk counts printed in Tables V and VI fix the rounding of
n_chunksRequired, the level count of Eq. (7) and the per-level split; the
invariant tests fix Eqs. (4)-(6) by what the quantities must satisfy.
"""
import json
import os

import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _tables():
    with open(os.path.join(GOLDEN, "magnus_chunk_tables.json")) as f:
        g = json.load(f)
    cases = []
    for name, n, pvc, h200 in g["suitesparse"]:
        cases.append((name, n, "PVC", pvc))
        cases.append((name, n, "H200", h200))
    for scale, pvc, h200 in g["rmat"]:
        if pvc is not None:
            cases.append((f"rmat{scale}", 1 << scale, "PVC", pvc))
        cases.append((f"rmat{scale}", 1 << scale, "H200", h200))
    return g["calibration"], cases


CAL, CASES = _tables()


def test_table_count():
    assert len(CASES) == 51


def _parse(entry: str):
    if ":" in entry:
        req, levels = entry.split(":")
        return int(req), [int(x) for x in levels.split(",")]
    return int(entry), [int(entry)]


@pytest.mark.parametrize("name,c_m,gpu,entry", CASES, ids=[f"{c[0]}-{c[2]}" for c in CASES])
def test_chunk_tables(name, c_m, gpu, entry):
    req, v = _parse(entry)
    p = oracle.magnus_params(c_m, dense_width=CAL[gpu]["dense_width"], n_chunks_max=CAL[gpu]["n_chunks_max"])
    assert p.n_chunks_required == req
    assert p.v_chunks == v
    assert p.n_levels == len(v)
    assert p.widths[-1] == CAL[gpu]["dense_width"]


@pytest.mark.parametrize("s_lm", [232448, 228 * 1024, 128 * 1024, 64 * 1024, 48 * 1024, 16 * 1024])
def test_param_invariants(s_lm):
    s_col, s_val, s_rp, s_h, s_bm, nsg = 4, 8, 8, 4, 1, 32
    p = oracle.magnus_params(1 << 20, s_lm=s_lm)
    # Eq. (4): alpha*tau slots of (key, value) fill at most s_LM bytes, one more tau would not.
    assert 2 * p.tau * (s_col + s_val) <= s_lm < 2 * (p.tau + 1) * (s_col + s_val)
    # Dense accumulator: value + bitmap byte per column, floored to a power of two.
    assert p.n_dense_numeric * (s_val + s_bm) <= s_lm < (p.n_dense_numeric + 1) * (s_val + s_bm)
    assert p.dense_width <= p.n_dense_numeric < 2 * p.dense_width
    assert p.dense_width & (p.dense_width - 1) == 0
    # Eq. (5): local arrays of the multisplit with n_chunksMax fit in s_LM, one more chunk would not.
    def eq5(ncm):
        return (s_h * (p.n_group_rows * nsg * ncm + 1) + s_rp * p.n_group_rows * ncm
                + (s_col + s_val) * p.n_min_group_elems)
    assert eq5(p.n_chunks_max_raw) <= s_lm < eq5(p.n_chunks_max_raw + 1)
    assert p.n_chunks_max <= p.n_chunks_max_raw < 2 * p.n_chunks_max
    # Half of s_LM holds the locally permuted elements; a group spans two rows at most.
    assert p.n_min_group_elems == s_lm // (2 * (s_col + s_val)) == p.tau
    assert p.n_group_rows == 2


def test_gb300_values():
    p = oracle.magnus_params(1 << 20)  # 227 KB per block on sm_103a
    assert (p.tau, p.dense_width, p.n_chunks_max) == (9685, 16384, 256)
    assert (p.n_chunks_required, p.n_levels, p.v_chunks, p.widths) == (64, 1, [64], [16384])
    p18 = oracle.magnus_params(1 << 18)
    assert (p18.n_chunks_required, p18.v_chunks) == (16, [16])
    p10 = oracle.magnus_params(1 << 10)
    assert (p10.n_chunks_required, p10.n_levels, p10.v_chunks) == (1, 0, [])


@pytest.mark.parametrize("c_m", [1, 2, 3, 1000, 4097, 65536, 65537, (1 << 20) + 1, 10 ** 7, 3 * 10 ** 9])
@pytest.mark.parametrize("d,ncm", [(16384, 256), (4096, 32), (8, 2), (1, 2), (64, 4)])
def test_levels_cover_columns(c_m, d, ncm):
    p = oracle.magnus_params(c_m, dense_width=d, n_chunks_max=ncm)
    prod = 1
    for v in p.v_chunks:
        assert 2 <= v <= ncm and v & (v - 1) == 0
        prod *= v
    assert prod == p.n_chunks_required
    # The chunks of the last level are D wide and together cover every column.
    assert d * p.n_chunks_required >= c_m
    assert p.n_chunks_required == 1 or d * p.n_chunks_required // 2 < c_m
    # Minimum number of levels: one fewer could not reach the required count.
    if p.n_levels >= 1:
        assert ncm ** (p.n_levels - 1) < p.n_chunks_required <= ncm ** p.n_levels
