"""The persistent GEMM's static tile deal, checked on the host.

The kernel walks its tiles with the same header (kth_tile) that this checker
compiles with g++: every tile of every problem must be dealt exactly once, a
launch of equal tiles must stay plain round robin over the whole launch, and
the catch-up phase must even out the launches that mix long and short tiles
(the FFN block's dA + dW2 launch: 16- and 64-block tiles).
"""
import os
import random
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
TILE_END = 6.0   # the per-tile cost the launcher adds to a tile's 128-wide blocks


@pytest.fixture(scope="module")
def checker(tmp_path_factory):
    gxx = shutil.which("g++")
    if gxx is None:
        pytest.skip("g++ not found")
    exe = str(tmp_path_factory.mktemp("deal") / "deal_check")
    subprocess.run([gxx, "-O2", "-std=c++17", "-o", exe, os.path.join(HERE, "deal_check.cpp")], check=True)

    def run(launches):
        text = "".join(f"{G} {len(probs)} " + " ".join(f"{n} {c}" for n, c in probs) + "\n" for G, probs in launches)
        out = subprocess.run([exe], input=text, capture_output=True, text=True, check=True).stdout.splitlines()
        assert len(out) == len(launches)
        res = []
        for line in out:
            f = line.split()
            assert f[0] == "ok", line
            plans = [tuple(map(int, f[4 + 3 * i: 7 + 3 * i])) for i in range((len(f) - 4) // 3)]
            res.append((float(f[1]), float(f[2]), float(f[3]), plans))
        return res

    return run


def test_every_tile_once_random(checker):
    rng = random.Random(20240611)
    launches = []
    for _ in range(400):
        G = rng.choice([1, 2, 3, 7, 64, 151, 152])
        probs = []
        for _ in range(rng.randint(1, 24)):
            n = rng.choice([0, 1, 2, G - 1 if G > 1 else 1, G, G + 1, rng.randint(0, 3000)])
            probs.append((n, float(rng.randint(1, 300)) + TILE_END))
        launches.append((G, probs))
    for mx, mrr, mean, plans in checker(launches):
        assert mx >= mean * (1 - 1e-9)


def test_equal_tiles_stay_round_robin(checker):
    # one problem, and several problems of one tile cost: the launch-wide round robin
    probs = [(1000, 22.0)], [(352, 70.0), (1408, 70.0), (77, 70.0), (5, 70.0)]
    for (mx, mrr, mean, plans), pr in zip(checker([(152, p) for p in probs]), probs):
        assert mx == mrr
        base = 0
        for (s, w, m), (n, _) in zip(plans, pr):
            assert (s, m) == (base % 152, 0)
            base += n


@pytest.mark.parametrize("name,probs,bound", [
    # d=2048, F=5632, T=8192: dW2 (F/128 x d/256 tiles over T/128 blocks), then dA (T/128 x F/256 tiles over d/128)
    ("dA+dW2 d2048", [(44 * 8, 64), (64 * 22, 16)], 1.05),
    # d=4096, F=14336, T=16384: dX (two terms over F), then dW1, dW3
    ("dX+dW1+dW3 d4096", [(128 * 16, 224), (32 * 56, 128), (32 * 56, 128)], 1.02),
])
def test_mixed_launch_balance(checker, name, probs, bound):
    (mx, mrr, mean, plans), = checker([(152, [(n, kb + TILE_END) for n, kb in probs])])
    assert mx <= mrr
    assert mx / mean <= bound, (name, mx / mean, mrr / mean)
