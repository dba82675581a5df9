"""Plant plausible mistakes in a copy of the oracle; the pins must catch each.

A mutant is built by a one-place text substitution in the oracle's source,
loaded as a fresh module, and run through every ``oracle_checks`` pin.  The
real oracle module is never modified.
"""

import os
import types

import pytest

import oracle.tide_oracle as real_oracle
import oracle_checks as C

SRC_PATH = real_oracle.__file__

MUTATIONS = {
    "landing sign": ("return (s - c) % L", "return (s + c) % L"),
    "relative index sign": ("return (n_dest - n_src) % M", "return (n_src - n_dest) % M"),
    "floor instead of ceil rows": ("r_pad = -(-shape[0] // N)", "r_pad = shape[0] // N + 1"),
    "rank-major uses piece size": ("return r * geo.S + geo.o[p]", "return r * geo.e[p] + geo.o[p]"),
    "param-major transposed": ("return geo.N * geo.o[p] + r * geo.e[p]",
                               "return r * geo.S + geo.o[p]"),
    "dropped local term": ("    for l in range(L):\n        acc1", "    for l in range(L - 1):\n        acc1"),
    "wrong sign at level 2": ("bsum = bsum + _node_partial", "bsum = bsum - _node_partial"),
    "source row index": ("src0 = r * e_p + a", "src0 = r * geo.Rp[p] + a"),
    "source rank transposed": ("return grads[src_rank][p][src0:src0 + count]",
                               "return grads[(src_rank % L) * M + src_rank // L][p][src0:src0 + count]"),
    "bf16 widening shift": ("<< np.uint32(16)).view", "<< np.uint32(15)).view"),
    "ascending node order": ("                        batch.append(n_src)\n        else:",
                             "                        batch.append(n_src)\n            batch.sort()\n        else:"),
    "flat level 2 across batches": ("                    acc2 = acc2 + bsum\n                out[o_p + a:o_p + b] = acc2",
                                    "                    acc2 = bsum\n                out[o_p + a:o_p + b] = acc2"),
    "slice length floor": ("return -(-S // L) if S > 0 else 0", "return S // L if S > 0 else 0"),
    "padding not zeroed": ("out[o_p + v:o_p + e_p] = np.float32(0.0)",
                           "out[o_p + v:o_p + e_p] = np.float32(1.0)"),
    "valid rows off by one": ("max(0, geo.rows[p] - r * geo.Rp[p])",
                              "max(0, geo.rows[p] - r * geo.Rp[p] + 1)"),
    # Starting either level alone at -0.0 changes nothing (the other level's
    # +0.0 absorbs it); starting both at the first term (-0.0 here) does.
    "accumulators start at first term": [
        ("acc1 = np.zeros(count, dtype=np.float32)", "acc1 = np.full(count, -0.0, dtype=np.float32)"),
        ("acc2 = np.zeros(b - a, dtype=np.float32)      # Reading R4",
         "acc2 = np.full(b - a, -0.0, dtype=np.float32)      # Reading R4"),
        ("bsum = np.zeros(b - a, dtype=np.float32)\n                    for n_src in batch:\n                        bsum = bsum + _node_partial",
         "bsum = np.full(b - a, -0.0, dtype=np.float32)\n                    for n_src in batch:\n                        bsum = bsum + _node_partial")],
    "recursive doubling sends 2^d": ("return min(2 ** d, M - 2 ** d)", "return 2 ** d"),
    "recursive doubling from the lower node": ("have[n] = have[n] + sent[(n + 2 ** d) % M]",
                                               "have[n] = have[n] + sent[(n - 2 ** d) % M]"),
    "stage slot rotated the wrong way": ("r = ((node + k) % M) * L + rail", "r = ((node - k) % M) * L + rail"),
    "landing stage adds a wrong source": ("c = b * L + (s - g) % L             # the batch's source",
                                          "c = b * L + (s + g) % L             # the batch's source"),
    "relative order descending": ("            for c in range(b * L, min(M, (b + 1) * L)):\n                batch +=",
                                  "            for c in reversed(range(b * L, min(M, (b + 1) * L))):\n                batch +="),
    "relative landing stage reads the wrong GPU": ("g = landing_gpu(s, c, L)            # where relative index",
                                                   "g = landing_gpu(s, c + 1, L)            # where relative index"),
    "unpadded all-gather keeps a padding row": ("return [params[p][:geo.rows[p] * geo.Kp[p]] for p in range(geo.P)]",
                                                "return [params[p][:(geo.rows[p] + 1) * geo.Kp[p]] for p in range(geo.P)]"),
    "inbox partial at the wrong landing GPU": ("                    g = landing_gpu(s, c, L)\n",
                                               "                    g = landing_gpu(s + 1, c, L)\n"),
    "accumulate drops the old value": ("x = (old[r] + x).astype(np.float32)", "x = (x + x).astype(np.float32)"),
    "single-element form without batches": ("        acc2 = np.float32(acc2 + bsum)", "        acc2 = np.float32(bsum)"),
    "average divides by M": ("x = (x / np.float32(geo.N)).astype(np.float32)",
                             "x = (x / np.float32(geo.N - 1 or 1)).astype(np.float32)"),
    "slot pack at op": ("slot[geo.N * geo.o[p]:geo.N * geo.o[p] + n] = grads[r][p][:n]",
                        "slot[geo.o[p]:geo.o[p] + n] = grads[r][p][:n]"),
    "AG piece offset": ("block[r * e_p:(r + 1) * e_p] = shards[r][o_p:o_p + e_p]",
                        "block[r * e_p:(r + 1) * e_p] = shards[(r + 1) % geo.N][o_p:o_p + e_p]"),
}


def _mutant(edits):
    with open(SRC_PATH) as f:
        src = f.read()
    for old, new in ([edits] if isinstance(edits, tuple) else edits):
        assert src.count(old) == 1, f"mutation anchor not unique: {old!r}"
        src = src.replace(old, new)
    mod = types.ModuleType("oracle_mutant")
    mod.__file__ = SRC_PATH
    exec(compile(src, SRC_PATH, "exec"), mod.__dict__)
    return mod


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_planted_mistake(name, monkeypatch):
    mutant = _mutant(MUTATIONS[name])
    monkeypatch.setattr(C, "O", mutant)
    caught = []
    for check in C.ALL_CHECKS:
        try:
            check()
        except Exception as exc:  # AssertionError or a crash both count as caught
            caught.append((check.__name__, type(exc).__name__))
    assert caught, f"no pin noticed the planted mistake {name!r}"


def test_unmutated_oracle_passes_all_pins():
    for check in C.ALL_CHECKS:
        check()
    assert os.path.exists(SRC_PATH)
