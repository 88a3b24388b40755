"""Plant plausible mistakes in a copy of the oracle's Python functions (cache
update, chunked prefill, latent expansion, DSA prefill scoring and top-k,
FP8 codecs) and check that the pins of that function catch each one (CPU
only).  The mistakes in the C core are planted by test_oracle_mutants.py."""
import os
import shutil
import subprocess
import sys

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)

# name: (pin file, original line(s), mutated line(s))
MUTANTS = {
    "appended values in reverse order": (
        "test_oracle_cache_pins.py",
        "v_out.append(np.concatenate([vc[b, :, :s], vn[b], vc[b, :, s + Tn:]], axis=1))",
        "v_out.append(np.concatenate([vc[b, :, :s], vn[b][:, ::-1], vc[b, :, s + Tn:]], axis=1))"),
    "chunk prefix shifted by one position": (
        "test_oracle_cache_pins.py",
        "k = np.concatenate([kc[:, :, :P], _f64(k_new)], axis=2)",
        "k = np.concatenate([kc[:, :, 1:P + 1], _f64(k_new)], axis=2)"),
    "cached decode drops the current token": (
        "test_oracle_cache_pins.py",
        "        if kn is not None:\n            kb = np.concatenate([kb, kn[b]], axis=1)",
        "        if kn is not None and False:\n            kb = np.concatenate([kb, kn[b]], axis=1)"),
    "shared key read from the front of the latent row": (
        "test_oracle_latent_pins.py",
        "lat, rope = c[:, :512], c[:, 512:]",
        "lat, rope = c[:, 64:], c[:, :64]"),
    "values built with W^K": (
        "test_oracle_latent_pins.py",
        'v = np.einsum("hdj,nj->hnd", wv, lat)',
        'v = np.einsum("hdj,nj->hnd", wk, lat)'),
    "prefill token cannot see its own position": (
        "test_oracle_dsa_prefill_pins.py",
        "mask = np.arange(Tk)[None, :] > (P + np.arange(Tq))[:, None]",
        "mask = np.arange(Tk)[None, :] >= (P + np.arange(Tq))[:, None]"),
    "prefill top-k ranks one future position": (
        "test_oracle_dsa_prefill_pins.py",
        "        n = P + i + 1\n",
        "        n = min(P + i + 2, Tk)\n"),
    "e4m3 scale for a 240 maximum": (
        "test_oracle_fp8_pins.py",
        "scale = (amax / np.float32(448.0)).astype(np.float32)",
        "scale = (amax / np.float32(240.0)).astype(np.float32)"),
    "record group scales reversed": (
        "test_oracle_fp8_pins.py",
        'rec[:, 512:528] = scale.astype("<f4").reshape(N, 4).view(np.uint8)',
        'rec[:, 512:528] = scale.astype("<f4").reshape(N, 4)[:, ::-1].copy().view(np.uint8)'),
    "index key scale not applied": (
        "test_oracle_fp8_pins.py",
        "k_deq = e4m3_values(k8) * _f64(kscale)[:, None]",
        "k_deq = e4m3_values(k8)"),
    "index query scale not applied": (
        "test_oracle_fp8_pins.py",
        "q_deq = (e4m3_values(qc) * qs.astype(np.float64)[:, None]).reshape(B, NH, D)",
        "q_deq = e4m3_values(qc).reshape(B, NH, D)"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, tmp_path):
    pin_file, old, new = MUTANTS[name]
    ign = shutil.ignore_patterns("_build", "__pycache__")
    shutil.copytree(os.path.join(ROOT, "oracle"), tmp_path / "oracle", ignore=ign)
    tests = tmp_path / "tests"
    tests.mkdir()
    for f in ("conftest.py", "test_oracle_pins.py", pin_file):
        shutil.copy(os.path.join(HERE, f), tests / f)
    shutil.copytree(os.path.join(HERE, "golden"), tests / "golden")
    init = tmp_path / "oracle" / "__init__.py"
    src = init.read_text()
    assert src.count(old) == 1, f"mutation site for '{name}' not found exactly once"
    init.write_text(src.replace(old, new))
    # the copy's conftest puts the copy's root (with the mutant oracle) first
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        str(tests / pin_file)],
                       cwd=tmp_path, capture_output=True, text=True, timeout=300)
    assert "passed" in r.stdout or "failed" in r.stdout or "error" in r.stdout.lower(), r.stdout
    assert r.returncode != 0, f"planted mistake '{name}' passed every pin of {pin_file}"


def test_unmutated_copy_passes(tmp_path):
    """The harness itself: the same copy without a planted mistake passes."""
    ign = shutil.ignore_patterns("_build", "__pycache__")
    shutil.copytree(os.path.join(ROOT, "oracle"), tmp_path / "oracle", ignore=ign)
    tests = tmp_path / "tests"
    tests.mkdir()
    files = sorted({m[0] for m in MUTANTS.values()})
    for f in ["conftest.py", "test_oracle_pins.py", *files]:
        shutil.copy(os.path.join(HERE, f), tests / f)
    shutil.copytree(os.path.join(HERE, "golden"), tests / "golden")
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-p", "no:cacheprovider",
                        *[str(tests / f) for f in files]],
                       cwd=tmp_path, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-2000:]
