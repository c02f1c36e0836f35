"""The seeded input generators (synthetic/generators.py): reproducible draws, one
stream per (seed, tensor name), the distributions the workloads state, and no
dependence on the oracle or the library (they only supply inputs)."""

import os

import numpy as np

from synthetic import generators as G

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_draws_are_reproducible_and_independent_of_call_order():
    a1 = G.packed_codes_uniform(64, 256, 3, "A")
    s1 = G.scales_uniform_normal(64, 256, 3, "SFA")
    s2 = G.scales_uniform_normal(64, 256, 3, "SFA")
    a2 = G.packed_codes_uniform(64, 256, 3, "A")
    assert np.array_equal(a1, a2) and np.array_equal(s1, s2)
    assert not np.array_equal(G.packed_codes_uniform(64, 256, 4, "A"), a1)       # another seed
    assert not np.array_equal(G.packed_codes_uniform(64, 256, 3, "B"), a1)       # another tensor
    assert np.array_equal(G.bf16_normal(8, 64, 1, "x"), G.bf16_normal(8, 64, 1, "x"))
    assert G.alpha_uniform(5) == G.alpha_uniform(5)


def test_distributions_match_the_workload_recipes():
    codes = G.packed_codes_uniform(256, 1024, 0, "A")
    nib = np.concatenate([codes & 15, codes >> 4]).ravel()
    counts = np.bincount(nib, minlength=16)
    assert counts.min() > 0.9 * nib.size / 16                          # all 16 codes, evenly
    sf = G.scales_uniform_normal(256, 1024, 0, "SFA")
    assert sf.min() == 0x18 and sf.max() == 0x58 and len(np.unique(sf)) == 65
    mix = G.scales_with_zero_and_subnormal(512, 1024, 0, "SFA")
    zero, sub = np.mean(mix == 0), np.mean((mix >= 1) & (mix <= 7))
    assert abs(zero - 0.05) < 0.01 and abs(sub - 0.05) < 0.01
    assert set(np.unique(mix[(mix > 7)])) <= set(range(0x18, 0x59))
    alphas = [G.alpha_uniform(s) for s in range(200)]
    assert 0.25 <= min(alphas) and max(alphas) <= 4.0
    x = G.bf16_normal(256, 256, 0, "x", 0.02)
    xf = (x.astype(np.uint32) << 16).view(np.float32)
    assert abs(float(xf.std()) - 0.02) < 0.002 and abs(float(xf.mean())) < 0.002


def test_generators_import_neither_the_oracle_nor_the_library():
    import ast

    tree = ast.parse(open(os.path.join(ROOT, "synthetic", "generators.py")).read())
    mods = set()
    for node in ast.walk(tree):
        if isinstance(node, ast.Import):
            mods |= {a.name.split(".")[0] for a in node.names}
        elif isinstance(node, ast.ImportFrom) and node.module:
            mods.add(node.module.split(".")[0])
    assert mods <= {"__future__", "hashlib", "numpy", "torch"}, mods
