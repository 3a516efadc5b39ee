"""Plant plausible mistakes in copies of the oracle and check a pin fails.

Each mutant is the oracle's C source with one textual change (a dropped
term, a wrong index, a swapped operand...), compiled on the CPU into a
temporary directory.  The committed oracle is never modified.
"""
import os

import pytest

import oracle_pins as P

MUTANTS = {
    "gqa_head_mapping": ("int32_t i = h * G + g;", "int32_t i = g * num_kv_heads + h;"),
    "scale_dropped": ("s[t] = scale * acc;", "s[t] = acc;"),
    "normalisation_dropped": ("o[d] = acc / denom;", "o[d] = acc;"),
    "exp_sign": ("s[t] = exp(s[t] - smax);", "s[t] = exp(smax - s[t]);"),
    "pv_reads_keys": ("acc += s[t] * V[", "acc += s[t] * K["),
    "query_head_index": ("q + ((int64_t)b * num_q_heads + i) * head_dim",
                         "q + ((int64_t)b * num_q_heads + h) * head_dim"),
    "gather_row_offset": ("(t % block_size)) * (int64_t)head_dim",
                          "((t + 1) % block_size)) * (int64_t)head_dim"),
    "gather_block_index": ("table_row[t / block_size]", "table_row[(t / block_size) / 2]"),
    "bf16_exponent_bias": ("e - 134);", "e - 133);"),
    "f16_subnormal_scale": ("ldexp((double)f, -24)", "ldexp((double)f, -25)"),
    "write_v_from_k": ("v_cache[dst + d] = v[src + d];", "v_cache[dst + d] = k[src + d];"),
    "write_row_reversed": ("* block_size + off) * (int64_t)head_dim",
                           "* block_size + (block_size - 1 - off)) * (int64_t)head_dim"),
    "negative_slot_written": ("if (s < 0) continue;", "if (s < 0) s = 0;"),
    "e4m3_exponent_bias": ("else mag = ldexp((double)(8 + f), e - 10);",
                           "else mag = ldexp((double)(8 + f), e - 9);"),
    "e4m3_round_up": ("double r = nearbyint(k);\n    if (r >= 8.0)", "double r = ceil(k);\n    if (r >= 8.0)"),
    "fp8_v_token_major": ("v_cache[((blk * num_kv_heads + h) * (int64_t)head_dim + d) * block_size + off] =",
                          "v_cache[((blk * num_kv_heads + h) * block_size + off) * (int64_t)head_dim + d] ="),
    "fp8_scale_not_applied": ("(double)k_scale[h];\n                V[", "1.0;\n                V["),
    "copy_v_from_k": ("v_cache[dst[i] * per_block + e] = v_cache[src[i] * per_block + e];",
                      "v_cache[dst[i] * per_block + e] = k_cache[src[i] * per_block + e];"),
    "prefill_diagonal_dropped": ("int32_t n_visible = pos + 1;", "int32_t n_visible = pos + 1 - (pos > 0);"),
    "prefill_position_base": ("int32_t pos = seq_lens[b] - piece_len + j;", "int32_t pos = j;"),
    "prefill_gqa_mapping": ("int32_t head = h * G + g;", "int32_t head = g * num_kv_heads + h;"),
    "prefill_rows_ignored": ("int64_t tok = rows ? rows[r] : r;", "int64_t tok = r;"),
    "prefill_query_row": ("q + (tok * num_q_heads + head) * (int64_t)head_dim;",
                          "q + ((int64_t)j * num_q_heads + head) * (int64_t)head_dim;"),
    "prefill_v_head": ("oracle_gather(v_cache, dtype, trow, n_visible, num_kv_heads, h,",
                       "oracle_gather(v_cache, dtype, trow, n_visible, num_kv_heads, 0,"),
    "copy_direction": ("k_cache[dst[i] * per_block + e] = k_cache[src[i] * per_block + e];",
                       "k_cache[src[i] * per_block + e] = k_cache[dst[i] * per_block + e];"),
}


SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle", "pa_oracle.c")


def _cases():
    """One mutant per (mistake, occurrence): a line the 16-bit and the FP8
    paths both contain is broken in each copy separately."""
    src = open(SRC).read()
    out = []
    for name in sorted(MUTANTS):
        n = src.count(MUTANTS[name][0])
        out += [(name, k) for k in range(max(n, 1))]
    return out


@pytest.mark.parametrize("name,occurrence", _cases(), ids=lambda v: str(v))
def test_some_pin_catches_mutant(oracle_mod, tmp_path, name, occurrence):
    src = open(SRC).read()
    old, new = MUTANTS[name]
    assert src.count(old) >= 1, f"mutation anchor for {name} missing from the oracle source"
    at = -1
    for _ in range(occurrence + 1):
        at = src.index(old, at + 1)
    mpath = tmp_path / f"mut_{name}_{occurrence}.c"
    mpath.write_text(src[:at] + new + src[at + len(old):])
    lib = oracle_mod.compile_source(str(mpath), str(tmp_path / f"mut_{name}_{occurrence}.so"))
    handle = oracle_mod.OracleLib(lib)
    caught = []
    for pin in P.ALL_PINS:
        try:
            pin(oracle_mod, handle=handle)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"no pin detects mutant {name}"


# Plausible mistakes in the dense (matrix-product) form of the prefill
# oracle, planted in a copy of its Python source.
PY_MUTANTS = {
    "dense_scale_dropped": ("S *= scale", "S *= 1.0"),
    "dense_mask_off_by_one": ("np.arange(hi)[None, :] > pos[rr][:, None]",
                              "np.arange(hi)[None, :] >= pos[rr][:, None]"),
    "dense_not_normalised": ("/ S.sum(axis=1, keepdims=True)", "/ 1.0"),
    "dense_gqa_mapping": ("i = h * G + g", "i = g * Hkv + h"),
    "dense_pv_reads_keys": ("(S @ V[:hi])", "(S @ K[:hi])"),
    "dense_position_base": ("pos = L - n + np.arange(n)", "pos = np.arange(n)"),
    "dense_last_key_dropped": ("hi = int(pos[rr[-1]]) + 1", "hi = int(pos[rr[-1]])"),
    "dense_max_not_subtracted": ("S -= S.max(axis=1, keepdims=True)", "S -= 0.0"),
}


@pytest.mark.parametrize("name", sorted(PY_MUTANTS))
def test_some_pin_catches_dense_mutant(oracle_mod, name):
    import inspect
    import textwrap
    import types
    src = textwrap.dedent(inspect.getsource(oracle_mod.prefill_dense))
    old, new = PY_MUTANTS[name]
    assert src.count(old) == 1, f"mutation anchor for {name} missing from prefill_dense"
    ns = dict(vars(oracle_mod))
    exec(compile(src.replace(old, new), f"<mutant {name}>", "exec"), ns)
    shim = types.SimpleNamespace(**{k: getattr(oracle_mod, k) for k in dir(oracle_mod)
                                    if not k.startswith("__")})
    shim.prefill_dense = ns["prefill_dense"]
    caught = []
    for pin in P.DENSE_PINS:
        try:
            pin(shim)
        except Exception:     # a failed check, or a mutant that cannot even run
            caught.append(pin.__name__)
    assert caught, f"no pin detects mutant {name}"
