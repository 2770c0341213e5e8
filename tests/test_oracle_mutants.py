"""Planted mistakes: each mutant is a copy of the oracle source with one
plausible error (a flipped sign, a wrong index, a dropped term, swapped
operands).  The test compiles it into a temporary directory, points the
oracle package at it and checks that at least one pin in
test_oracle_pins.py fails.  The real oracle is never modified."""
import functools
import os
import subprocess

import pytest

import oracle as O
from tests import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(O.__file__), "pie_oracle.cpp")

MUTANTS = {
    "rope_sign": [("out[i] = x[i] * c - x[i + h] * s;", "out[i] = x[i] * c + x[i + h] * s;"),
                  ("out[i + h] = x[i + h] * c + x[i] * s;", "out[i + h] = x[i + h] * c - x[i] * s;")],
    "rope_freq": [("-2.0 * i / d", "-1.0 * i / d")],
    "rope_pairing": [("out[i] = x[i] * c - x[i + h] * s;", "out[i] = x[i] * c - x[h - 1 - i] * s;")],
    "kv_swap": [("load(D.dtype, v_pool, vb + j)", "load(D.dtype, k_pool, vb + j)")],
    "scale": [("1.0 / std::sqrt(static_cast<double>(d))", "1.0 / static_cast<double>(d)")],
    "gqa_map": [("const int g = h / G;", "const int g = h % Hkv;")],
    "causal_off_by_one": [("return s <= M.slots[r];", "return s < M.slots[r];")],
    "mask_bit_order": [("(words[base + (s >> 5)] >> (s & 31)) & 1u",
                        "(words[base + (s >> 5)] >> (31 - (s & 31))) & 1u")],
    "kv_len_bound": [("for (int s = 0; s < M.kv_len[l]; ++s)", "for (int s = 0; s <= M.kv_len[l]; ++s)"),
                     ("if (s >= M.kv_len[l]) return false;", "")],
    "lse_drops_max": [("L = m + std::log(sum);", "L = std::log(sum);")],
    "page_table_lane_offset": [("int page = M.page_ids[M.page_indptr[l] + s / D.page_size];",
                                "int page = M.page_ids[s / D.page_size];")],
    "page_offset": [("* D.page_size + s % D.page_size) *", "* D.page_size + (s + 1) % D.page_size) *")],
    "fold_no_clamp": [("k = c < 0 ? 0 : (c > n ? n : c);", "k = c;")],
    "fold_all_off_by_one": [("case ORC_FOLD_ALL: k = n; break;", "case ORC_FOLD_ALL: k = n - 1; break;")],
    "frozen_check": [("if (s < frozen_len[l]) {", "if (s <= frozen_len[l]) {")],
    "bf16_truncates": [("std::nearbyint(a / quantum)", "std::floor(a / quantum)")],
    "v_rotated_dropped_memcpy": [("std::memcpy(static_cast<char*>(v_pool) + dst * eb,",
                                  "std::memcpy(static_cast<char*>(k_pool) + dst * eb,")],
    "dup_target_check": [("if (t[i] == t[i - 1]) return ORC_EINVAL;", ";")],
    "default_readout_first_row": [("out[R] = M.row_indptr[l + 1] - 1;", "out[R] = M.row_indptr[l];")],
}

def _expand(fn):
    """A pin function, or one partial per parameter set of a parametrized pin."""
    marks = [m for m in getattr(fn, "pytestmark", []) if m.name == "parametrize"]
    if not marks:
        return [fn]
    names, values = marks[0].args[0], marks[0].args[1]
    out = []
    for val in values:
        args = val if "," in names else (val,)
        out.append(functools.partial(fn, *args))
    return out


PIN_FUNCS = [f for n in sorted(dir(pins)) if n.startswith("test_")
             for f in _expand(getattr(pins, n))]


def _build(tmp_path, name, edits):
    src = open(SRC).read()
    for old, new in edits:
        assert old in src, (name, old)
        src = src.replace(old, new)
    cpp = tmp_path / f"{name}.cpp"
    cpp.write_text(src)
    so = tmp_path / f"lib{name}.so"
    subprocess.check_call(["g++", "-O1", "-std=c++17", "-fPIC", "-shared", "-o", str(so),
                           str(cpp), "-lpthread"])
    return str(so)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_fails_a_pin(name, tmp_path, monkeypatch):
    so = _build(tmp_path, name, MUTANTS[name])
    monkeypatch.setattr(O, "_lib", O.load(so))
    caught = None
    for f in PIN_FUNCS:
        try:
            f()
        except Exception:  # an assertion or a numeric error both count as caught
            caught = getattr(f, "__name__", getattr(getattr(f, "func", None), "__name__", "?"))
            break
    assert caught is not None, f"mutant {name} passed every pin"


def test_unmutated_copy_passes_every_pin(tmp_path, monkeypatch):
    so = _build(tmp_path, "clean", [])
    monkeypatch.setattr(O, "_lib", O.load(so))
    for f in PIN_FUNCS:
        f()
