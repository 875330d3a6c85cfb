"""Plant plausible mistakes in copies of the oracle and check that the pins see them.

Every mutant below is a one-line edit of ``oracle/oracle.c`` compiled into a
throw-away library (CPU only; nothing here touches a GPU).  A mutant that no
pin rejects would mean the pins leave that part of the oracle unchecked.
"""
import os
import shutil

import pytest

import oracle
from oracle_pins import ALL_PINS

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")
HDR = os.path.join(os.path.dirname(oracle.__file__), "oracle.h")

MUTANTS = {
    # RMSNorm
    "eps_outside_sqrt": ("sqrt(ss / (double)D + eps)", "sqrt(ss / (double)D) + eps"),
    "mean_over_D_minus_1": ("ss / (double)D + eps", "ss / (double)(D - 1) + eps"),
    "weight_wrong_index": ("* r * orc_bf16_value(w[i])", "* r * orc_bf16_value(w[i % 64])"),
    "weight_dropped": ("* r * orc_bf16_value(w[i])", "* r"),
    # RoPE
    "rope_sign": ("n[a] = na * c - nb * s;", "n[a] = na * c + nb * s;"),
    "rope_dropped_term": ("n[b] = nb * c + na * s;", "n[b] = nb * c;"),
    "rope_cos_sin_swapped": ("double c = (double)cs[i], s = (double)cs[half + i];",
                             "double s = (double)cs[i], c = (double)cs[half + i];"),
    "neox_partner_index": ("int b = neox ? off + i + half", "int b = neox ? off + i + 1"),
    "interleaved_as_neox": ("int a = neox ? off + i : off + 2 * i;", "int a = off + i;"),
    "dsv4_rope_offset": ("DSV4_ROPE_OFF = 448,", "DSV4_ROPE_OFF = 384,"),
    # partial rotation (positions in the pins stay far enough from the end of
    # the table that the widened reads stay inside it)
    "partial_rotates_whole_head": ("rope_rotate(n, mg, 0, A->rot, A->neox, cs);",
                                   "rope_rotate(n, mg, 0, A->D, A->neox, cs);"),
    "partial_table_stride": ("const float* cs = A->cs + pos * A->rot;",
                             "const float* cs = A->cs + pos * (A->rot / 2);"),
    "qk_q_k_weights_swapped": ("h < A->Hq ? A->qw : A->kw", "h < A->Hk ? A->qw : A->kw"),
    "qk_v_not_copied": ("  if (out != in)\n    memcpy(", "  if (0)\n    memcpy("),
    # codecs
    "bf16_truncates": ("nearbyint(a / spacing)", "trunc(a / spacing)"),
    "bf16_precision": ("ldexp(1.0, e - 7)", "ldexp(1.0, e - 8)"),
    "e4m3_ties_away": ("else c = (lo % 2 == 0) ? lo : hi;", "else c = hi;"),
    "e4m3_bias": ("ldexp(8.0 + mf, ef - 10)", "ldexp(8.0 + mf, ef - 11)"),
    "ue8m0_no_correction": ("int e = k - 9; /* 448", "int e = k - 9; return e; /* 448"),
    "ue8m0_uses_512": ("while (ldexp(448.0, e) < amax) ++e;", "while (ldexp(512.0, e) < amax) ++e;"),
    "ue8m0_bias": ("int b = e + 127;", "int b = e + 128;"),
    # DSV4 entry
    "scale_offset": ("DSV4_SCALE_AT = 576", "DSV4_SCALE_AT = 575"),
    "rope_bytes_big_endian": ("entry[DSV4_ROPE_AT + 2 * i] = (uint8_t)(bits & 0xff);",
                              "entry[DSV4_ROPE_AT + 2 * i] = (uint8_t)(bits >> 8);"),
    "amax_wrong_block": ("if (fabs(blk[j]) > amax) amax = fabs(blk[j]);",
                         "if (fabs(blk[j + 1]) > amax) amax = fabs(blk[j + 1]);"),
    "codes_unscaled": ("orc_e4m3_encode(ldexp(blk[j], -e))", "orc_e4m3_encode(blk[j])"),
    "codes_rounded_via_fp32": ("orc_e4m3_encode(ldexp(blk[j], -e))",
                               "orc_e4m3_encode((double)(float)ldexp(blk[j], -e))"),
    "amax_rounded_to_fp32": ("const uint8_t byte = orc_ue8m0_byte(amax);",
                             "const uint8_t byte = orc_ue8m0_byte((double)(float)amax);"),
    # the comparison's excusal inputs: magnitude sums and exponent margins
    "mag_ignores_table": ("mag[a] = fabs(na * c) + fabs(nb * s);", "mag[a] = fabs(na) + fabs(nb);"),
    "mag_partner_swapped": ("mag[b] = fabs(nb * c) + fabs(na * s);",
                            "mag[b] = fabs(na * c) + fabs(nb * s);"),
    "mag_unrotated_dims": ("      for (int i = 0; i < D; ++i) mg[i] = fabs(n[i]);",
                           "      for (int i = 0; i < D; ++i) mg[i] = 2.0 * fabs(n[i]);"),
    "margin_zero": ("  return up < dn ? up : dn;", "  return 0.0;"),
    "margin_one_side": ("  return up < dn ? up : dn;", "  return up;"),
    "margin_wrong_boundary": ("const double dn = 1.0 - ldexp(448.0, e - 1) / amax;",
                              "const double dn = 1.0 - ldexp(448.0, e - 2) / amax;"),
    # (kept inside the cache: a mutant must not write out of bounds)
    "slot_hardcoded_block": ("(blk * A->block_size + off)", "((blk * 64 + off) % A->num_slots)"),
    "skip_ignored": ("const int64_t s = A->slot[t];", "const int64_t s = A->slot[t] < 0 ? 0 : A->slot[t];"),
    "gather_scale_bias": ("const int ex = (int)e[DSV4_SCALE_AT + b] - 127;",
                          "const int ex = (int)e[DSV4_SCALE_AT + b] - 126;"),
    "gather_block_scale": ("const int ex = (int)e[DSV4_SCALE_AT + b] - 127;",
                           "const int ex = (int)e[DSV4_SCALE_AT] - 127;"),
    "kv_uses_q_weight": ("rms_norm_weight(A->kv + krow, A->kvw,", "rms_norm_weight(A->kv + krow, A->qw,"),
}


@pytest.fixture(scope="module")
def mutant_dir(tmp_path_factory):
    return tmp_path_factory.mktemp("oracle_mutants")


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_reject_mutant(name, mutant_dir):
    old, new = MUTANTS[name]
    text = open(SRC).read()
    assert text.count(old) == 1, f"mutation site for {name} not unique/present"
    d = mutant_dir / name
    d.mkdir()
    shutil.copy(HDR, d / "oracle.h")
    (d / "oracle.c").write_text(text.replace(old, new))
    so = oracle.build(force=True, src=str(d / "oracle.c"), out=str(d / "liboracle.so"))
    L = oracle.load_variant(so)
    failed = []
    try:
        for pin in ALL_PINS:
            try:
                pin(L)
            except Exception as e:  # noqa: BLE001 -- any failure counts as detection
                failed.append((pin.__name__, type(e).__name__))
                break
    finally:
        oracle.unload_variant(L)
    assert failed, f"no pin detects mutant {name}"
