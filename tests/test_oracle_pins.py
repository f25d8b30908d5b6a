"""The oracle against its pins, and planted mistakes in the oracle against the same pins.

CPU only.  A planted mistake is a textual change to a copy of one oracle source file, executed
as a fresh module on the CPU; the real oracle files are never modified.
"""

import os
import types

import numpy as np
import pytest

import oracle
import pins

ORACLE_DIR = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle")


@pytest.mark.parametrize("check", pins.ALL_CHECKS, ids=lambda c: c.__name__)
def test_oracle_passes_pin(check):
    check(oracle)


def _load(name, replace=None):
    with open(os.path.join(ORACLE_DIR, name + ".py")) as f:
        src = f.read()
    if replace is not None:
        old, new = replace
        assert old in src, f"mutation target {old!r} not found in oracle/{name}.py"
        src = src.replace(old, new)
    mod = types.ModuleType(f"mutant_{name}")
    exec(compile(src, f"mutant_{name}.py", "exec"), mod.__dict__)
    return mod


def _mutant(file, old, new):
    mods = {n: _load(n, (old, new) if n == file else None)
            for n in ("attention", "layouts", "ulysses", "backward")}
    ns = types.SimpleNamespace()
    for n in ("attention", "merge"):
        setattr(ns, n, getattr(mods["attention"], n))
    for n in ("shard_positions", "sub_chunk_positions", "visible_pair_count"):
        setattr(ns, n, getattr(mods["layouts"], n))
    for n in ("seq_to_head", "head_to_seq"):
        setattr(ns, n, getattr(mods["ulysses"], n))
    for n in ("attention_backward", "chunk_backward"):
        setattr(ns, n, getattr(mods["backward"], n))
    return ns


MUTANTS = [
    # (id, file, original text, planted mistake)
    ("gqa_mod_mapping", "attention", "k[:, h // group, :]", "k[:, h % hkv, :]"),
    ("dropped_scale", "attention", "s = scale * (q[rr, h, :] @ kh.T)", "s = (q[rr, h, :] @ kh.T)"),
    ("k_for_v", "attention", "(e @ vh)", "(e @ kh)"),
    ("exclusive_diagonal", "attention", "k_pos[None, :] <= q_pos[rr][:, None]",
     "k_pos[None, :] < q_pos[rr][:, None]"),
    ("reversed_causality", "attention", "k_pos[None, :] <= q_pos[rr][:, None]",
     "k_pos[None, :] >= q_pos[rr][:, None]"),
    ("lse_log2", "attention", "m + np.log(np.where(has, z, 1.0)), -np.inf)\n    return out, lse",
     "m + np.log2(np.where(has, z, 1.0)), -np.inf)\n    return out, lse"),
    ("lse_missing_max", "attention", "lse[b0:b0 + len(rr), h] = np.where(has, m + np.log(",
     "lse[b0:b0 + len(rr), h] = np.where(has, 0 * m + np.log("),
    ("merge_sum_not_max", "attention", "m = lse.max(axis=0)", "m = lse.sum(axis=0)"),
    ("merge_unnormalised", "attention", "num / np.where(has, z, 1.0)[..., None]",
     "num / 1.0"),
    ("merge_lse_no_shift", "attention", "out_lse = np.where(has, m + np.log(",
     "out_lse = np.where(has, np.log("),
    ("strided_row_major", "layouts", "rank + cp * i", "rank * local_len + i"),
    ("contiguous_start", "layouts", "start = rank * local_len", "start = rank * cp"),
    ("visible_strict", "layouts", 'side="right"', 'side="left"'),
    ("two_block_mirror", "layouts", "late = [(2 * cp - 1 - rank) * block + i",
     "late = [(cp + rank) * block + i"),
    ("balanced_by_tokens", "layouts", "need = r * total  # compare b (b + 1) cp against this",
     "need = r * seq_len * seq_len  # compare b (b + 1) cp against this"),
    ("balanced_off_by_one", "layouts", "        while b * (b + 1) * cp < need:\n            b += 1\n        bounds.append(b)",
     "        while b * (b + 1) * cp < need:\n            b += 1\n        bounds.append(b + 1)"),
    ("bwd_no_softmax_jacobian_term", "backward",
     "ds = p * (dp - (p * dp).sum(axis=1, keepdims=True))", "ds = p * dp"),
    ("bwd_dq_unscaled", "backward", "dq[:, h, :] = scale * (ds @ k[:, g, :])",
     "dq[:, h, :] = (ds @ k[:, g, :])"),
    ("bwd_dk_uses_p", "backward", "dk[:, g, :] += scale * (ds.T @ q[:, h, :])",
     "dk[:, g, :] += scale * (p.T @ q[:, h, :])"),
    ("bwd_gqa_overwrite", "backward", "dv[:, g, :] += p.T @ d_o[:, h, :]",
     "dv[:, g, :] = p.T @ d_o[:, h, :]"),
    ("bwd_dv_uses_v", "backward", "dp = d_o[:, h, :] @ v[:, g, :].T", "dp = d_o[:, h, :] @ k[:, g, :].T"),
    ("chunk_delta_from_chunk_only", "backward", "ds = p * (dp - delta[:, h][:, None])",
     "ds = p * (dp - (p * dp).sum(axis=1, keepdims=True))"),
    ("chunk_lse_ignored", "backward",
     "p = np.exp(s - np.where(finite, lse[:, h], 0.0)[:, None])", "p = np.exp(s)"),
    ("ulysses_interleaved_q_heads", "ulysses",
     "out[r][np.asarray(positions[s])] = x_shards[s][:, r * hl:(r + 1) * hl, :]",
     "out[r][np.asarray(positions[s])] = x_shards[s][:, r::cp, :]"),
    ("ulysses_local_order", "ulysses",
     "out[r][np.asarray(positions[s])] = x_shards[s][:, r * hl:(r + 1) * hl, :]",
     "out[r][s * local:(s + 1) * local] = x_shards[s][:, r * hl:(r + 1) * hl, :]"),
]


@pytest.mark.parametrize("mid,file,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistake(mid, file, old, new):
    mutant = _mutant(file, old, new)
    failed = []
    for check in pins.ALL_CHECKS:
        try:
            with np.errstate(all="ignore"):
                check(mutant)
        except (AssertionError, ValueError, IndexError, FloatingPointError):
            failed.append(check.__name__)
    assert failed, f"no pin catches the planted mistake {mid}"


def test_unmutated_copy_passes():
    # the loader itself does not break anything
    ns = _mutant("attention", "_ROW_BLOCK = 64", "_ROW_BLOCK = 3")
    for check in pins.ALL_CHECKS:
        check(ns)
