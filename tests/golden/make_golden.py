"""Writes tests/golden/oracle_vectors.json: small encoder / decoder / all-gather
decode vectors computed by the CPU oracle alone (inputs are seeded numpy draws
made here).  They freeze the oracle's outputs so that a later change of its
arithmetic shows up as a diff; every change must name the passage, or the
reading of it, that justifies it.  The pages print no worked numeric example,
so no fixture here is a page value.

    python tests/golden/make_golden.py
"""
import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))
import oracle as O  # noqa: E402

CASES = [  # (bits, block, rounding, ef, hadamard, n, dtype)
    (1, 8, 0, True, 0, 40, "f32"), (2, 32, 1, True, 0, 200, "f32"), (4, 128, 0, True, 0, 300, "bf16"),
    (4, 64, 1, False, 0, 129, "f32"), (8, 16, 0, True, 0, 100, "bf16"), (12, 32, 1, True, 0, 96, "f32"),
    (16, 8, 0, True, 0, 33, "f32"), (4, 128, 0, True, 32, 256, "f32"), (8, 256, 1, True, 64, 512, "bf16"),
]


def bf16_bits(x):
    u = x.view(np.uint32).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


def exact_fraction_case():
    """Stochastic rounding at the exact fraction: 2-bit codes, blocks of 8 with
    scale 1 (each holds a 1.0).  Where an element's u = (r mod 2^23) 2^-23 lies in
    (1/2, 3/4), its value is t = u - 1 + d for d = 2^-25, 0, -2^-25 in turn:
    the fraction t - floor(t) = 1 + t is u + 2^-25, u, u - 2^-25, so q = 0, -1, -1
    (rounding 1 + t to fp32 would give a tie that goes to u itself for d = 2^-25,
    and q = -1).  expect_q lists those positions and their q."""
    seed, n = 5, 1024
    words = O.random_words(seed, 0, 0, n)
    m = words & 0x7FFFFF
    x = np.zeros(n, np.float32)
    expect = []
    used = set()
    for h in np.nonzero((m > 1 << 22) & (m < 3 << 21))[0]:
        h = int(h)
        b0 = h // 8 * 8
        if b0 in used:
            continue
        used.add(b0)
        d = (2.0 ** -25, 0.0, -2.0 ** -25)[len(expect) % 3]
        t = float(m[h]) * 2.0 ** -23 + d - 1.0
        assert float(np.float32(t)) == t
        x[b0 + (h - b0 + 4) % 8] = 1.0
        x[h] = t
        expect.append((h, 0 if d > 0 else -1))
        if len(expect) == 9:
            break
    p = O.params(2, 8, O.SR, seed=seed)
    codes, scales = O.quantize_pack(x, p)
    mean = O.unpack_dequant(codes, scales, n, p, 0.5, O.BF16)
    return {"bits": 2, "block": 8, "rounding": 1, "ef": False, "hadamard": 0, "n": n, "dtype": "f32",
            "seed": seed, "index_offset": 0, "x": x.tobytes().hex(),
            "err_in": np.zeros(n, np.float32).tobytes().hex(), "codes": codes.tobytes().hex(),
            "scales": scales.tobytes().hex(), "err_out": None, "mean_bf16": mean.tobytes().hex(),
            "expect_q": expect}


def main():
    out = []
    for k, (bits, block, rnd, ef, H, n, dt) in enumerate(CASES):
        rng = np.random.default_rng(1000 + k)
        x = (rng.standard_t(3, n) * 1e-2).astype(np.float32)
        xin = x if dt == "f32" else bf16_bits(x)
        e = (rng.standard_normal(n) * 1e-3).astype(np.float32)
        p = O.params(bits, block, rnd, seed=77 + k, index_offset=4 * k, hadamard=H)
        e_out = e.copy() if ef else None
        codes, scales = O.quantize_pack(xin, p, e_out)
        mean = O.unpack_dequant(codes, scales, n, p, 0.5, O.BF16)
        out.append({"bits": bits, "block": block, "rounding": rnd, "ef": ef, "hadamard": H, "n": n,
                    "dtype": dt, "seed": 77 + k, "index_offset": 4 * k,
                    "x": xin.tobytes().hex(), "err_in": e.tobytes().hex(),
                    "codes": codes.tobytes().hex(), "scales": scales.tobytes().hex(),
                    "err_out": e_out.tobytes().hex() if ef else None,
                    "mean_bf16": mean.tobytes().hex()})
    out.append(exact_fraction_case())
    # a W=3 decoder case on the first three encodings' formats (4-bit, block 128)
    rng = np.random.default_rng(7)
    n = 384
    enc = [O.quantize_pack((rng.standard_normal(n) * 1e-2).astype(np.float32), O.params(4, 128))
           for _ in range(3)]
    e2 = (rng.standard_normal(n) * 1e-3).astype(np.float32)
    e2_out = e2.copy()
    s, co, so = O.unpack_dequant_reduce_requant([c for c, _ in enc], [q for _, q in enc], n, O.params(4, 128),
                                                True, e2_out, O.params(4, 128, 1, seed=5, philox_stream=1))
    dec = {"n": n, "codes_in": [c.tobytes().hex() for c, _ in enc], "scales_in": [q.tobytes().hex() for _, q in enc],
           "err2_in": e2.tobytes().hex(), "sum": s.tobytes().hex(), "codes_out": co.tobytes().hex(),
           "scales_out": so.tobytes().hex(), "err2_out": e2_out.tobytes().hex()}
    with open(os.path.join(HERE, "oracle_vectors.json"), "w") as f:
        json.dump({"encoder": out, "decoder": dec}, f, indent=1)
        f.write("\n")


if __name__ == "__main__":
    main()
