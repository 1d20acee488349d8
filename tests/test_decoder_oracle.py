"""The oracle's decoder composition against its pins, and planted mistakes that the pins
must catch (CPU only)."""
import importlib.util
import os

import pytest

import oracle
from oracle import decoder as odec
import decoder_pins

SOURCE = os.path.join(os.path.dirname(oracle.SOURCE), "decoder.py")

# Plausible mistakes in composing the decoder, each a single textual change.
MUTATIONS = {
    "k_and_v_slices_swapped": (
        "k = _bf16(O.rope(qkv[:, H:H + Hkv].copy(), pos, rope_base))\n        v = qkv[:, H + Hkv:]",
        "k = _bf16(O.rope(qkv[:, H + Hkv:].copy(), pos, rope_base))\n        v = qkv[:, H:H + Hkv]"),
    "q_taken_after_kv": ("q = _bf16(O.rope(qkv[:, :H].copy(), pos, rope_base))",
                         "q = _bf16(O.rope(qkv[:, 2 * Hkv:].copy(), pos, rope_base))"),
    "rope_on_v_too": ("v = qkv[:, H + Hkv:]",
                      "v = _bf16(O.rope(qkv[:, H + Hkv:].copy(), pos, rope_base))"),
    "rope_not_on_k": ("k = _bf16(O.rope(qkv[:, H:H + Hkv].copy(), pos, rope_base))",
                      "k = qkv[:, H:H + Hkv]"),
    "positions_from_one": ("pos = np.arange(L)", "pos = np.arange(1, L + 1)"),
    "attention_not_causal": ("causal=True, q_offset=0", "causal=False, q_offset=0"),
    "attention_residual_dropped": ("h = _bf16(h + _bf16(O.linear(att, f(lw[\"wo\"]))[0]))",
                                   "h = _bf16(O.linear(att, f(lw[\"wo\"]))[0])"),
    "mlp_residual_dropped": ("h = _bf16(h + _bf16(O.linear(a, f(lw[\"wdown\"]))[0]))",
                             "h = _bf16(O.linear(a, f(lw[\"wdown\"]))[0])"),
    "norm_weights_swapped": ("n = _bf16(O.rmsnorm(h, f(lw[\"ln1\"]), eps))",
                             "n = _bf16(O.rmsnorm(h, f(lw[\"ln2\"]), eps))"),
    "final_norm_dropped": ("n = _bf16(O.rmsnorm(h, f(weights[\"lnf\"]), eps))", "n = h"),
    "attention_output_not_rounded": ("att = _bf16(att[0].transpose(1, 0, 2).reshape(L, H * D))",
                                     "att = att[0].transpose(1, 0, 2).reshape(L, H * D)"),
    "heads_flattened_in_wrong_order": (
        "att = _bf16(att[0].transpose(1, 0, 2).reshape(L, H * D))",
        "att = _bf16(att[0].transpose(1, 2, 0).reshape(L, H * D))"),
}


def _load_variant(tmp_path, name, old, new):
    src = open(SOURCE).read()
    assert src.count(old) == 1, "mutation anchor must occur once: %s" % name
    src = src.replace(old, new).replace("from . import default", "from oracle import default")
    path = tmp_path / ("decoder_%s.py" % name)
    path.write_text(src)
    spec = importlib.util.spec_from_file_location("decoder_%s" % name, str(path))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


@pytest.mark.parametrize("pin", decoder_pins.DECODER_PINS, ids=lambda p: p.__name__)
def test_decoder_oracle_pin(pin):
    pin(odec)


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_decoder_mutation_is_caught(name, tmp_path):
    old, new = MUTATIONS[name]
    mod = _load_variant(tmp_path, name, old, new)
    caught = []
    for pin in decoder_pins.DECODER_PINS:
        try:
            pin(mod)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, "decoder mutation %s was not caught by any pin" % name
