"""Plant plausible mistakes in a copy of the oracle and check that the pins catch each.

The copy is compiled into a temporary library; the shipped oracle is never
modified.  Each mutant must disagree with at least one pin: the library
conv3d special case, the chunked == whole invariant with its cache contents,
or the closed-form constant-input count.
"""
import os

import numpy as np
import pytest

import oracle
from tests.test_oracle_pins import torch_reference

MUTANTS = {
    "flipped_kernel_w": ("const int ws = w + dw - pw;", "const int ws = w + (kw - 1 - dw) - pw;"),
    "future_frames": ("const int ts = t + dt - (kt - 1);", "const int ts = t - dt;"),
    "no_bias": ("if (c->b) v += c->b[co];", "(void)0;"),
    "no_residual": ("if (c->r) v += c->r[o];", "(void)0;"),
    "transposed_spatial_taps": ("(((size_t)co * kt + dt) * kh + dh) * kw + dw)",
                                "(((size_t)co * kt + dt) * kh + dw) * kw + dh)"),
    "no_spatial_padding_shift": ("const int ph = (kh - 1) / 2, pw = (kw - 1) / 2;",
                                 "const int ph = 0, pw = 0;"),
    "dropped_channel": ("for (int ci = 0; ci < Cin; ++ci)", "for (int ci = 1; ci < Cin; ++ci)"),
    "cache_from_front": ("memcpy(cache_out, xe + frame * Tc,", "memcpy(cache_out, xe,"),
    "replicate_first_frame_history": ("memset(xe, 0, sizeof(double) * frame * P); /* zero history */",
                                      "for (int q = 0; q < P; ++q) memcpy(xe + frame * q, x_chunk, sizeof(double) * frame);"),
    "chunk_reads_one_frame_late": ("const int te = t + dt;", "const int te = t + dt + (dt < kt - 1);"),
}


def pins_hold(lib: oracle.OracleLib) -> bool:
    rng = np.random.default_rng(123)
    T, H, W, Cin, Cout = 6, 4, 5, 3, 2
    x = rng.standard_normal((T, H, W, Cin))
    w = rng.standard_normal((Cout, 3, 3, 3, Cin))
    b = rng.standard_normal(Cout)
    r = rng.standard_normal((T, H, W, Cout))
    ref = torch_reference(x, w, b, r)
    tol = 1e-11
    if not np.allclose(lib.conv_whole(x, w, b, r), ref, rtol=0, atol=tol):
        return False
    for parts in ([6], [2, 1, 3], [1, 1, 4], [5, 1]):
        y, caches = lib.conv_chunked(x, w, b, r, chunks=parts)
        if not np.allclose(y, ref, rtol=0, atol=tol):
            return False
        end = 0
        for p, cache in zip(parts, caches):
            end += p
            for j in range(2):
                src = end - 2 + j
                exp = x[src] if src >= 0 else np.zeros_like(x[0])
                if not np.array_equal(cache[j], exp):
                    return False
    ones = lib.conv_whole(np.ones((4, 3, 3, 2)), np.ones((1, 3, 3, 3, 2)))
    for t in range(4):
        for h in range(3):
            for ww in range(3):
                n = 2 * min(t + 1, 3) * (3 - (h == 0) - (h == 2)) * (3 - (ww == 0) - (ww == 2))
                if ones[t, h, ww, 0] != n:
                    return False
    return True


def test_unmodified_oracle_passes_the_pin_suite():
    assert pins_hold(oracle.OracleLib(oracle.build()))


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(oracle.SOURCE).read()
    assert old in src, "mutation anchor not found: %s" % name
    mutated = tmp_path / "mutant.c"
    mutated.write_text(src.replace(old, new))
    lib = oracle.OracleLib(oracle.compile_source(str(mutated), str(tmp_path / "libmutant.so")))
    assert not pins_hold(lib), "planted mistake %r went unnoticed" % name
