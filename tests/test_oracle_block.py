"""The attention-block oracle against its pins, and planted mistakes in copies
of its source that the pins must catch. CPU only."""
import importlib.util

import pytest

import oracle_block_pins as P
from oracle import attn_block as OB


@pytest.mark.parametrize("pin", P.ALL_BLOCK_PINS, ids=lambda f: f.__name__)
def test_block_oracle_pin(pin):
    pin(OB)


MUTATIONS = {
    "unbiased_variance": ("var = ((x - mean) ** 2).mean(axis=-1, keepdims=True)",
                          "var = ((x - mean) ** 2).sum(axis=-1, keepdims=True) / (x.shape[-1] - 1)"),
    "eps_dropped": ("np.sqrt(var + eps)", "np.sqrt(var)"),
    "gain_and_bias_swapped": ("* np.asarray(gamma, np.float64) + np.asarray(beta, np.float64)",
                              "* np.asarray(beta, np.float64) + np.asarray(gamma, np.float64)"),
    "qkv_bias_dropped": ("linear(n.reshape(B * S, hidden), w_qkv, b_qkv)", "linear(n.reshape(B * S, hidden), w_qkv, None)"),
    "k_v_swapped": ("k = qkv[..., Hq * D: (Hq + Hkv) * D]", "k = qkv[..., (Hq + Hkv) * D:]"),
    "not_causal_exact": ("            if causal:\n                i = np.arange", "            if False:\n                i = np.arange"),
    "not_causal_held": ("kind = _oracle.MASK_CAUSAL if causal else _oracle.MASK_NONE", "kind = _oracle.MASK_NONE"),
    "attention_output_unrounded": ("    a = hold(a, hold_in)\n", "\n"),
    "scale_without_sqrt": ("scale=1.0 / math.sqrt(D))", "scale=1.0 / D)"),
    "residual_dropped": (".reshape(B, S, hidden) + x\n", ".reshape(B, S, hidden)\n"),
    "kv_group_modulo": ("k[b, :, h // g, :].T", "k[b, :, h % Hkv, :].T"),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_in_block_oracle_is_caught(name, tmp_path):
    src = open(OB.__file__).read()
    old, new = MUTATIONS[name]
    assert src.count(old) == 1, f"anchor of {name} not found exactly once"
    path = tmp_path / "attn_block_mutant.py"
    path.write_text(src.replace(old, new))
    spec = importlib.util.spec_from_file_location("attn_block_mutant", path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    caught = []
    for pin in P.ALL_BLOCK_PINS:
        try:
            pin(mod)
        except (AssertionError, ValueError):
            caught.append(pin.__name__)
    assert caught, f"no pin caught {name}"
