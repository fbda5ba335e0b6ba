"""tune.py's table writer (CPU only): a partial sweep replaces exactly the
rows it measured, keeps the fastest variant per (op, direction, dtype, M
bucket, N), leaves every other row and the default rows as they were, and is
stable; a small-M measurement gets a row of its own ahead of the any-M row;
a near tie keeps the current variant."""
import os
import re
import shutil

from rmsnorm_norm_fwd_gb300 import tune

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
TABLE = os.path.join(ROOT, "rmsnorm_norm_fwd_gb300", "csrc", "dispatch_table.inc")


def _rows(text):
    start = text.index("// ---- measured rows (tune.py) ----")
    end = text.index("// ---- forward defaults")
    return [l for l in text[start:end].splitlines() if l.startswith("{")]


def test_emit_merges_partial_sweep(tmp_path):
    path = tmp_path / "dispatch_table.inc"
    shutil.copy(TABLE, path)
    before = path.read_text()
    old_rows = _rows(before)
    results = [  # two variants for one measured shape, one for a new N (small M)
        {"op": "ln", "dir": 1, "dtype": "bf16", "M": 16384, "N": 8192, "variant": "slow", "gbs": 100.0},
        {"op": "ln", "dir": 1, "dtype": "bf16", "M": 16384, "N": 8192, "variant": "fast", "gbs": 200.0},
        {"op": "rms", "dir": 0, "dtype": "fp16", "M": 8, "N": 24, "variant": "tiny", "gbs": 1.0},
    ]
    tune.emit(results, str(path))
    after = path.read_text()
    new_rows = _rows(after)
    # the measured LN row now names the faster variant; N = 8192 bf16 is 1024 vectors
    assert any(r.startswith('{1, 1, 2, -1, 1024, "fast"}') for r in new_rows)
    assert not any('"slow"' in r for r in new_rows)
    # a new (op, dir, dtype, M bucket, N) is added (24 fp16 elements = 3
    # vectors; 8 rows: the small-M bucket)
    assert any(r.startswith(f'{{0, 0, 1, {tune.SMALL_M}, 3, "tiny"}}') for r in new_rows)
    # every other measured row is unchanged
    key = lambda r: tuple(re.match(r"\{(\d+), (\d+), (\d+), (-?\d+), (\d+),", r).groups())
    untouched = {key(r): r for r in old_rows
                 if key(r) not in {("1", "1", "2", "-1", "1024"), ("0", "0", "1", str(tune.SMALL_M), "3")}}
    new_by_key = {key(r): r for r in new_rows}
    for k, r in untouched.items():
        assert new_by_key[k] == r
    assert len(new_rows) == len(old_rows) + 1
    # the defaults after the measured block are untouched
    tail = lambda t: t[t.index("// ---- forward defaults"):]
    assert tail(after) == tail(before)
    # emitting nothing changes nothing
    tune.emit([], str(path))
    assert path.read_text() == after


def test_small_m_row_precedes_any_m_row(tmp_path):
    path = tmp_path / "dispatch_table.inc"
    shutil.copy(TABLE, path)
    tune.emit([{"op": "rms", "dir": 1, "dtype": "bf16", "M": 1024, "N": 1024, "variant": "small", "gbs": 9.0},
               {"op": "rms", "dir": 1, "dtype": "bf16", "M": 65536, "N": 1024, "variant": "big", "gbs": 99.0}],
              str(path))
    rows = _rows(path.read_text())
    i_small = next(i for i, r in enumerate(rows) if '"small"' in r)
    i_big = next(i for i, r in enumerate(rows) if '"big"' in r)
    assert i_small < i_big
    assert rows[i_small].startswith(f'{{0, 1, 2, {tune.SMALL_M}, 128, "small"}}')
    assert rows[i_big].startswith('{0, 1, 2, -1, 128, "big"}')


def test_near_tie_keeps_the_current_variant(tmp_path):
    """A measured row keeps its variant unless a challenger is faster by more
    than KEEP_MARGIN (event timestamps step by about 2 us, so short calls tie)."""
    path = tmp_path / "dispatch_table.inc"
    shutil.copy(TABLE, path)
    rows = _rows(path.read_text())
    # the LayerNorm forward bf16 row at N = 131072 (16384 vectors), any M
    row = next(r for r in rows if r.startswith("{1, 0, 2, -1, 16384,"))
    current = re.search(r'"([^"]+)"', row).group(1)
    base = {"op": "ln", "dir": 0, "dtype": "bf16", "M": 2048, "N": 131072}
    near = 1000.0 * (1 + tune.KEEP_MARGIN / 2)
    tune.emit([dict(base, variant=current, gbs=1000.0), dict(base, variant="challenger", gbs=near)], str(path))
    row = next(r for r in _rows(path.read_text()) if r.startswith("{1, 0, 2, -1, 16384,"))
    assert f'"{current}"' in row
    far = 1000.0 * (1 + 2 * tune.KEEP_MARGIN)
    tune.emit([dict(base, variant=current, gbs=1000.0), dict(base, variant="challenger", gbs=far)], str(path))
    row = next(r for r in _rows(path.read_text()) if r.startswith("{1, 0, 2, -1, 16384,"))
    assert '"challenger"' in row
