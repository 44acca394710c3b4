"""Planted mistakes in copies of the oracle must each be caught by some pin (no GPU).

Each case rewrites one expression of oracle/w4a16_oracle.c in a temporary copy -- a dropped
term, a wrong sign, a shifted index, a transposed or reversed operand -- compiles it, and runs
every pin against it.  The real oracle is never modified.  All mutations keep memory accesses
in bounds so a broken copy cannot crash the test process.
"""
import os

import pytest

import oracle
import pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "w4a16_oracle.c")

MUTATIONS = [
    ("sign of q - zp", "return (q - zp) * s;", "return (zp - q) * s;"),
    ("u4b8 bias 7", "? 8.0 : orc_h16(zeros[(long)g * n + col], bf16);",
     "? 7.0 : orc_h16(zeros[(long)g * n + col], bf16);"),
    ("nibble order high first", "return (int)((word >> (4 * (row % 8))) & 0xFu);",
     "return (int)((word >> (4 * (7 - row % 8))) & 0xFu);"),
    ("group off by one row", "    return row / group_size;\n}",
     "    return (row > 0 ? row - 1 : 0) / group_size;\n}"),
    ("scale column reversed", "double s = orc_h16(scales[(long)g * n + col], bf16);",
     "double s = orc_h16(scales[(long)g * n + (n - 1 - col)], bf16);"),
    ("zero point column dropped", "? 8.0 : orc_h16(zeros[(long)g * n + col], bf16);",
     "? 8.0 : orc_h16(zeros[(long)g * n], bf16);"),
    ("g_idx ignored", "    if (g_idx)\n        return g_idx[row];\n", "\n"),
    ("dropped accumulation", "acc[j] += av * wr[j];", "acc[j] = av * wr[j];"),
    ("W band column shifted", "jb->weight_type, row, c0 + j, jb->bf16);",
     "jb->weight_type, row, c0 + (j + 1) % width, jb->bf16);"),
    ("A reversed along K", "double av = orc_h16(jb->a[(long)i * jb->lda + row], jb->bf16);",
     "double av = orc_h16(jb->a[(long)i * jb->lda + (jb->k - 1 - row)], jb->bf16);"),
    ("bf16 activations read as fp16", "double av = orc_h16(jb->a[(long)i * jb->lda + row], jb->bf16);",
     "double av = orc_h16(jb->a[(long)i * jb->lda + row], 0);"),
    ("bf16 exponent bias", "v = ldexp(1.0 + frac / 128.0, expo - 127);", "v = ldexp(1.0 + frac / 128.0, expo - 126);"),
    ("bf16 fraction width", "v = ldexp(1.0 + frac / 128.0, expo - 127);", "v = ldexp(1.0 + frac / 64.0, expo - 127);"),
    ("half exponent bias", "v = ldexp(1.0 + frac / 1024.0, expo - 15);",
     "v = ldexp(1.0 + frac / 1024.0, expo - 14);"),
    ("half subnormal scale", "v = ldexp((double)frac, -24);", "v = ldexp((double)frac, -23);"),
    ("tile nibble placement", "word |= code << (4 * p + 16 * e);",
     "word |= code << (4 * (2 * p + e));"),
    ("tile row pairing", "int sorted_row = kb * 64 + h * 32 + 2 * j + 8 * p + e;",
     "int sorted_row = kb * 64 + h * 32 + 8 * j + 2 * p + e;"),
    ("tile half order", "out[base + h * 512 + c * 4 + j] = (int32_t)word;",
     "out[base + (1 - h) * 512 + c * 4 + j] = (int32_t)word;"),
    ("csr pair ids", "ex_pairs[cursor[selected[p]]++] = p;", "ex_pairs[cursor[selected[p]]++] = pair_tok[p];"),
    ("csr offsets", "ex_off[active] = (int32_t)cursor[e];", "ex_off[active] = (int32_t)cursor[e + 1];"),
    ("qzeros plus one dropped", "zero_points[(long)g * n + col] = (double)raw + 1.0;",
     "zero_points[(long)g * n + col] = (double)raw;"),
    ("group count ignores divisibility", "group_size % 16 != 0 || k % group_size != 0",
     "group_size % 16 != 0"),
    ("fp8 dropped accumulation", "acc[j] += a_ik * wrow[j];", "acc[j] = a_ik * wrow[j];"),
    ("e4m3 exponent bias", "v = ldexp(1.0 + frac / 8.0, expo - 7);", "v = ldexp(1.0 + frac / 8.0, expo - 8);"),
    ("e4m3 subnormal scale", "v = ldexp((double)frac / 8.0, -6);", "v = ldexp((double)frac / 8.0, -7);"),
    ("fp8 byte order", "return (int)((word >> (8 * (row % 4))) & 0xFFu);",
     "return (int)((word >> (8 * (3 - row % 4))) & 0xFFu);"),
    ("fp8 tile quarter and word swapped", "int row = kb * 64 + 16 * q + 4 * t + i;", "int row = kb * 64 + 16 * t + 4 * q + i;"),
    ("moe sentinel off by one", "sorted_ids[len + r] = n_ids; /* the sentinel */",
     "sorted_ids[len + r] = n_ids - 1; /* the sentinel */"),
    ("moe top-k weight dropped", "double w = topk_weights ? (double)topk_weights[id] : 1.0;", "double w = 1.0;"),
    ("moe A row by id", "orc_gemm(a + (long)(id / top_k) * lda, lda, 1,", "orc_gemm(a + (long)(id % m) * lda, lda, 1,"),
    ("silu sign of exp", "return x / (1.0 + exp(-x));", "return x / (1.0 + exp(x));"),
    ("gelu cubic constant", "(x + 0.044715 * x * x * x)", "(x + 0.44715 * x * x * x)"),
    ("glu operands swapped", "h[i] = orc_act(gate[i], kind) * up[i];", "h[i] = orc_act(up[i], kind) * gate[i];"),
    ("by-groups scale dropped", "c[(long)i * n + j] += orc_half_to_double(scales[(long)g * n + j]) * t[j];",
     "c[(long)i * n + j] += t[j];"),
]


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_mutation_is_caught(tmp_path, name, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor not unique/present: {old!r}"
    mutated = tmp_path / "mutant.c"
    mutated.write_text(src.replace(old, new))
    lib = oracle.build(force=True, src=str(mutated), out=str(tmp_path / "libmutant.so"))
    orc = oracle.Oracle(lib)
    failures = [p.__name__ for p in pins.ALL_PINS if p(orc) is not None]
    assert failures, f"no pin caught the planted mistake: {name}"
