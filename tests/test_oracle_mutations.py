"""Mutation check of the oracle pins.

Each case plants one plausible mistake in a scratch copy of the oracle, on the
CPU only.  The pins in test_oracle_pins.py must then fail.  A mutation that
survives means some part of the oracle is effectively unpinned.
"""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

MUTATIONS = [
    ("floor instead of half-even rint", "np.rint(t)", "np.floor(t)"),
    ("2^b levels instead of 2^b - 1", "levels = F32(2 ** bits - 1)", "levels = F32(2 ** bits)"),
    ("INT4 scale without the 16x", "scale.astype(np.float64) * 16.0", "scale.astype(np.float64) * 1.0"),
    ("top-k score without the zero-point term",
     "return ((Sf * unit).astype(F32) + beta).astype(F32)", "return (Sf * unit).astype(F32)"),
    ("top-k zero-point products summed as a running fp32 sum",
     "    Z = int(np.sum(np.rint(p.astype(np.float64) * (2.0 ** (Z_BITS - f))).astype(np.int64)))",
     "    Z = float(np.sum(p, dtype=np.float32)) * 2.0 ** (Z_BITS - f)"),
    ("top-k zero-point products rounded at 2^-20 instead of 2^-40", "Z_BITS = 40", "Z_BITS = 20"),
    ("INT4 midpoint at 7 instead of 8", "MID_NIBBLE = 8", "MID_NIBBLE = 7"),
    ("INT4 midpoint zero point left unmoved in the top-k score",
     "        z = (z + (F32(MID_NIBBLE) * s).astype(F32)).astype(F32)", "        z = z"),
    ("1-bit centred levels at a half of the range instead of a quarter", "CENTER_SHIFT = 0.25", "CENTER_SHIFT = 0.5"),
    ("1-bit centred reading without the halved scale", '"int1c": ("int1", 1, 0.5),', '"int1c": ("int1", 1, 1),'),
    ("1-bit centred zero point left unmoved in the top-k score",
     "        z = (z + (F32(CENTER_SHIFT) * s).astype(F32)).astype(F32)", "        z = z"),
    ("causal offset off by one", "nvis = (P - gamma + i + 1) if P else 0", "nvis = (P - gamma + i) if P else 0"),
    ("strided instead of consecutive GQA grouping", "hq = h * hg + hh", "hq = hh * H + h"),
    ("flush one token early", "if self.r == 2 * self.G:", "if self.r == 2 * self.G - 1:"),
    ("ties won by the higher index", "key=lambda t: (-float(sc[t]), t))[:k]", "key=lambda t: (-float(sc[t]), -t))[:k]"),
    ("reversed code order within a byte", "out |= (c[..., e] << (pb * e)).astype(np.uint8)",
     "out |= (c[..., per - 1 - e] << (pb * e)).astype(np.uint8)"),
    ("values quantized per channel instead of per token",
     "c, s, z = quantize_minmax(x, bits, axis=-1)", "c, s, z = quantize_minmax(x, bits, axis=-2)"),
    ("fetch lets the -1 padding wrap to the last row", "                if 0 <= t < N:\n                    sel_k",
     "                if t < N:\n                    sel_k"),
    ("fetch takes the value row from the key store", "sel_v[b, h, j] = full_v[b, h, t]", "sel_v[b, h, j] = full_k[b, h, t]"),
]


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_pins_catch_planted_mistake(tmp_path, name, old, new):
    for sub in ("oracle", "tests"):
        shutil.copytree(os.path.join(ROOT, sub), tmp_path / sub,
                        ignore=shutil.ignore_patterns("__pycache__"))
    shutil.copy(os.path.join(ROOT, "kvq_inputs.py"), tmp_path / "kvq_inputs.py")
    src = tmp_path / "oracle" / "kvq_oracle.py"
    text = src.read_text()
    assert old in text, f"mutation anchor not found: {old}"
    src.write_text(text.replace(old, new))
    r = subprocess.run([sys.executable, "-m", "pytest", "tests/test_oracle_pins.py", "-x", "-q",
                        "-p", "no:cacheprovider"], cwd=tmp_path, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"planted mistake '{name}' was not caught by any pin"
