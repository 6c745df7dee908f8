"""The oracle against its pins, and the pins against planted mistakes (CPU only)."""
import os
import subprocess
import sys

import numpy as np
import pytest

import oracle
import workloads
from tests import oracle_pins, parity


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(orc, pin):
    pin(orc)


# Each planted mistake is a plausible slip in oracle.c; at least one pin must fail on it.
MUTATIONS = [
    ("relu_dropped", "double relu = a > 0.0 ? a : 0.0;", "double relu = a;"),
    ("relu_on_wrong_side", "double a = scale * dot[h];", "double a = dot[h];"),
    ("weight_sign", "s += w[h] * relu;", "s -= w[h] * relu;"),
    ("q_transposed", "qr[h * ORACLE_DIM + i]", "qr[i * ORACLE_HEADS + h]"),
    ("page_index", "page_table[(int64_t)req * pt_stride + t / ORACLE_PAGE]",
     "page_table[(int64_t)req * pt_stride + t % ORACLE_PAGE]"),
    ("slot_index", "int64_t slot = t % ORACLE_PAGE;", "int64_t slot = t / ORACLE_PAGE;"),
    ("scale_dropped", "return (double)k_scale[page * ORACLE_PAGE + slot];", "return 1.0;"),
    ("scale_logical", "return (double)k_scale[page * ORACLE_PAGE + slot];",
     "return (double)k_scale[t];"),
    ("e4m3_bias", "exp_field - 7);", "exp_field - 8);"),
    ("e4m3_subnormal", "ldexp((double)man_field / 8.0, 1 - 7)", "ldexp((double)man_field / 8.0, -7)"),
    ("bf16_shift", "((uint32_t)bits) << 16", "((uint32_t)bits) << 15"),
    ("bound_inclusive", "if (t1 > row_bound[r]) t1 = row_bound[r];",
     "if (t1 > row_bound[r] + 1) t1 = row_bound[r] + 1;"),
    ("row_request", "row_query(q_bf16, w, r, qt, wd);\n                cur_row = r;\n            }\n            for",
     "row_query(q_bf16, w, r, qt, wd);\n                cur_row = r;\n            }\n            if (0) for"),
    ("ties_high_index", "if (x->pos < y->pos) return -1;\n    if (x->pos > y->pos) return 1;",
     "if (x->pos < y->pos) return 1;\n    if (x->pos > y->pos) return -1;"),
    ("ascending", "if (x->score > y->score) return -1;\n    if (x->score < y->score) return 1;",
     "if (x->score > y->score) return 1;\n    if (x->score < y->score) return -1;"),
    ("no_padding", "(j < n) ? v[j].pos : -1", "(j < n) ? v[j].pos : 0"),
    ("radix_negative", "return (u >> 31) ? ~u : (u | 0x80000000u);", "return (u >> 31) ? u : (u | 0x80000000u);"),
    ("negative_zero", "if (x == 0.0f) x = 0.0f;", ""),
    ("digit_shift", "oracle_radix_key(scores[(int64_t)r * ld + t]) >> 26", "oracle_radix_key(scores[(int64_t)r * ld + t]) >> 25 & 63"),
    ("top1_ties_high_index", "if (v > bv) {", "if (v >= bv) {"),
    ("top1_nan_kept", "const float v = isnan(row[j]) ? -1e30f : row[j];", "const float v = row[j];"),
    ("top1_first_nan_kept", "float bv = isnan(row[0]) ? -1e30f : row[0];", "float bv = row[0];"),
    ("encode_truncates", "double m = rint(ldexp(a, 3 - e));", "double m = floor(ldexp(a, 3 - e));"),
    ("encode_bias", "(uint8_t)((e + 7) << 3)", "(uint8_t)((e + 8) << 3)"),
    ("encode_subnormal_step", "const double m = rint(ldexp(a, 9));", "const double m = rint(ldexp(a, 8));"),
    ("key_scale_unscaled", "const float sc = amax > 0.0f ? amax / 448.0f : 1.0f;", "const float sc = amax > 0.0f ? amax : 1.0f;"),
    ("new_key_page_by_slot", "*page = page_table[(int64_t)row_req[r] * pt_stride + t / ORACLE_PAGE];",
     "*page = page_table[(int64_t)row_req[r] * pt_stride + t % ORACLE_PAGE];"),
    ("new_key_slot_by_page", "*slot = t % ORACLE_PAGE;", "*slot = t / ORACLE_PAGE;"),
    ("new_key_at_bound", "const int64_t t = (int64_t)row_bound[r] - 1;", "const int64_t t = (int64_t)row_bound[r];"),
    ("new_key_row_as_request", "page_table[(int64_t)row_req[r] * pt_stride + t / ORACLE_PAGE]",
     "page_table[(int64_t)r * pt_stride + t / ORACLE_PAGE]"),
    ("new_key_for_bound_zero", "    if (row_bound[r] == 0) return 0;\n", ""),
    ("merge_offset_dropped", "v[n].pos = part_idx[at] + offset[s];", "v[n].pos = part_idx[at];"),
    ("merge_empty_entries_kept", "if (part_idx[at] < 0) continue;", ""),
    ("merge_no_padding", "out_idx[(int64_t)r * K + j] = j < n ? v[j].pos : -1;",
     "out_idx[(int64_t)r * K + j] = j < n ? v[j].pos : 0;"),
    ("merge_part_stride", "const int64_t at = ((int64_t)s * R + r) * Kin + j;", "const int64_t at = ((int64_t)r * S + s) * Kin + j;"),
]


# Mistakes that read or write past a buffer on every input; the pins see the crash.
CAUGHT_BY_CRASH_ONLY = set()

_RUN_PINS = """
import sys
sys.path.insert(0, {root!r})
import oracle
from tests import oracle_pins
mutant = oracle.Oracle({lib!r})
for pin in oracle_pins.ALL_PINS:
    try:
        pin(mutant)
    except (AssertionError, ValueError):
        print("FAILED_PIN", pin.__name__, flush=True)
print("DONE", flush=True)
"""


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_pins_reject_planted_mistake(tmp_path, name, old, new):
    """Every planted mistake fails a pin.  Each mutant runs in its own process, since
    a mistake in indexing may also read out of bounds; a mutant that crashes before
    any pin has failed counts as caught only by the crash, and is listed as such."""
    src = oracle.source_text()
    assert src.count(old) == 1, f"mutation anchor for {name} not found exactly once"
    lib = oracle.compile_variant(src.replace(old, new), str(tmp_path / f"liboracle_{name}.so"))
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    proc = subprocess.run([sys.executable, "-c", _RUN_PINS.format(root=root, lib=lib)],
                          capture_output=True, text=True, timeout=600)
    failed = [x.split()[1] for x in proc.stdout.splitlines() if x.startswith("FAILED_PIN ")]
    if name in CAUGHT_BY_CRASH_ONLY:
        assert proc.returncode != 0 or failed
        return
    assert failed, f"no pin caught the planted mistake {name} (exit {proc.returncode})"


def test_page_test_shapes_fixture():
    path = os.path.join(os.path.dirname(__file__), "golden", "page_test_shapes.txt")
    fields = {}
    for line in open(path):
        line = line.split("[")[0].strip()
        if not line or line.startswith("#"):
            continue
        k, v = line.split("=")
        fields[k.strip()] = [int(x) for x in v.split()]
    pos, rows = workloads.page_positions()
    assert fields["topk_positions"] == pos and fields["topk_rows"] == rows
    assert fields["top_k"] == [workloads.TOPK]
    assert fields["first_digit_shift"] == [26] and fields["first_digit_bins"] == [64]


def test_page_position_bounds(orc):
    """The page's smallest top-k position (bound 8448) at its row counts, checked by
    brute force selection and the structural invariants."""
    pos, rows = workloads.page_positions()
    b = pos[0] + 1
    for n in rows:
        p = workloads.build("pos", [b], [n], "e4m3", seed=20 + n)
        s = orc.score(p)
        s32 = s.astype(np.float32)
        idx = orc.topk(s32, p.row_bound, workloads.TOPK)
        parity.check_index_rows(idx, p.row_bound, workloads.TOPK)
        parity.check_order(idx, s32, p.row_bound, workloads.TOPK)
        assert np.all(np.isfinite(s[np.arange(n)[:, None], np.arange(b - n + 1)[None, :]]))


def test_endtoend_rule_rejects_far_swap(orc):
    """The allowed-swap rule accepts a swap at the k-th value and rejects a far one."""
    rng = np.random.default_rng(3)
    ref = np.sort(rng.standard_normal(100))[::-1].copy()[None, :] * 8
    ref[0, 9] = ref[0, 10] - 1e-4                     # near-tie across the k = 10 boundary
    s32 = ref.astype(np.float32)
    O = orc.topk(s32, np.array([100], np.int32), 10)
    G = O.copy()
    G[0, 9] = 10 if O[0, 9] == 9 else 9               # swap the near-tied pair
    parity.check_endtoend(G, ref, O, np.array([100]), 10)
    bad = O.copy()
    bad[0, 0] = 99                                    # the lowest score instead of the top
    with pytest.raises(AssertionError):
        parity.check_endtoend(bad, ref, O, np.array([100]), 10)
