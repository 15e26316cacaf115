"""8-bit pixel output of the narrow head (the device half of the asynchronous frame output path).

Two checks:
* against the oracle: oracle.quantize_u8 of the exact (fp64) convolution.  The GPU accumulates in
  fp32, so its pixel can differ from the exact value's pixel only where the exact value lies
  within the accumulation error of a point where the pixel changes (a bf16 rounding tie that
  moves the value across a pixel boundary); there it may differ by one level, everywhere else it
  must be equal;
* against the same plan's bf16 output, quantised on the host: exactly equal (both from the same
  accumulation, so the integer decision is taken on the same value), and bit-identical across
  chunkings.
"""
import numpy as np
import pytest
import torch

import chunked_causal_convolution_gb300 as cc3d
import oracle
from tests.helpers import run_chunks, small_inputs, to_device, to_f64

# a bound on |fp32 accumulation - exact| for these layers (K = 27 * Cin <= 2592 products of
# bf16 values, sums of order RMS(y)): about 1e-6 * RMS is typical, this leaves a wide margin
ACC_BOUND = 2e-4

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


def quant_u8(y_bf16: torch.Tensor) -> np.ndarray:
    """clamp(rint((v + 1) * 127.5), 0, 255) in fp32 with one rounding per operation."""
    v = y_bf16.float().cpu().numpy().astype(np.float32)
    t = (v + np.float32(1.0)) * np.float32(127.5)
    return np.clip(np.rint(t), 0, 255).astype(np.uint8)


def run_chunks_u8(plan, x, w, b, r, chunks):
    caches = [plan.new_cache(x.device), plan.new_cache(x.device)]
    ys, s = [], 0
    for k, c in enumerate(chunks):
        ys.append(plan.forward_chunk_u8(x[s:s + c], w, b, r[s:s + c] if r is not None else None,
                                        caches[k % 2] if k else None, caches[(k + 1) % 2]))
        s += c
    return torch.cat(ys)


@pytest.mark.parametrize("Cin,Cout,T,H,W,chunks,residual", [
    (96, 3, 5, 6, 130, [2, 3], True),
    (32, 1, 4, 9, 300, [1, 3], False),
])
def test_u8_head_equals_quantised_bf16_output(Cin, Cout, T, H, W, chunks, residual):
    raw = small_inputs(Cin, Cout, T, H, W, "bf16", 77 + Cout, bias=True, residual=residual)
    dev = {k: to_device(v, "bf16") for k, v in raw.items()}
    plan = cc3d.CausalConv3dPlan(Cin, Cout, H, W)
    assert plan.kernel == "tc_bf16_head"
    y, _ = run_chunks(plan, dev["x"], dev["w"], dev["b"], dev.get("r"), chunks)
    yu8 = run_chunks_u8(plan, dev["x"], dev["w"], dev["b"], dev.get("r"), chunks)
    assert plan.status() == 0
    assert yu8.dtype == torch.uint8 and yu8.shape == y.shape
    exp = quant_u8(y)
    got = yu8.cpu().numpy()
    assert np.array_equal(got, exp), int((got != exp).sum())
    # against the oracle
    ref = oracle.conv_whole(to_f64(raw["x"], "bf16"), to_f64(raw["w"], "bf16"), to_f64(raw["b"], "bf16"),
                            to_f64(raw["r"], "bf16") if residual else None)
    q_ref = oracle.quantize_u8(ref)
    diff = np.abs(got.astype(np.int64) - q_ref.astype(np.int64))
    assert diff.max() <= 1, int(diff.max())
    # quantize_u8 is monotone in y, so a GPU value within delta of the exact one gives a pixel in
    # [Q(y - delta), Q(y + delta)]; where those agree the pixel is decided and must be equal
    delta = ACC_BOUND * float(np.sqrt(np.mean(ref ** 2)))
    lo, hi = oracle.quantize_u8(ref - delta), oracle.quantize_u8(ref + delta)
    assert np.all((lo <= got) & (got <= hi)), int(((lo > got) | (got > hi)).sum())
    decided = lo == hi
    assert decided.mean() > 0.9, decided.mean()
    assert np.array_equal(got[decided], q_ref[decided])
    # the outputs (about N(0, 1), with the residual N(0, 2)) reach both clamps and the interior
    assert (exp == 0).any() and (exp == 255).any() and ((exp > 0) & (exp < 255)).mean() > 0.25
    for alt in ([T], [1] * T):
        assert torch.equal(run_chunks_u8(plan, dev["x"], dev["w"], dev["b"], dev.get("r"), alt), yu8)
    plan.close()


def _u8_cases(n=12, seed=818):
    rng = np.random.RandomState(seed)
    out = []
    for _ in range(n):
        T = int(rng.randint(2, 8))
        cuts = sorted(rng.choice(np.arange(1, T), size=rng.randint(0, min(3, T - 1) + 1), replace=False))
        b1 = [0] + [int(x) for x in cuts] + [T]
        cuts2 = sorted(rng.choice(np.arange(1, T), size=rng.randint(0, min(3, T - 1) + 1), replace=False))
        b2 = [0] + [int(x) for x in cuts2] + [T]
        out.append(dict(Cin=int(rng.choice([32, 64, 96, 128])), Cout=int(rng.randint(1, 6)), T=T,
                        H=int(rng.randint(1, 10)), W=int(rng.choice([int(rng.randint(1, 140)), 256, 300])),
                        residual=bool(rng.randint(2)),
                        chunks=[[b - a for a, b in zip(b1, b1[1:])], [b - a for a, b in zip(b2, b2[1:])]]))
    return out


U8_CASES = _u8_cases()


@pytest.mark.parametrize("c", U8_CASES, ids=["%dto%d_T%d_%dx%d%s" % (c["Cin"], c["Cout"], c["T"], c["H"], c["W"],
                                                                      "_r" if c["residual"] else "") for c in U8_CASES])
def test_random_u8_heads_against_the_oracle_and_every_chunking(c):
    """Random narrow heads and chunkings: the 8-bit pixels are bit-identical across chunkings,
    equal to the plan's bf16 output quantised on the host, and inside the oracle's monotone
    bounds."""
    raw = small_inputs(c["Cin"], c["Cout"], c["T"], c["H"], c["W"], "bf16", 300 + c["T"] + c["W"], bias=True,
                       residual=c["residual"])
    dev = {k: to_device(v, "bf16") for k, v in raw.items()}
    plan = cc3d.CausalConv3dPlan(c["Cin"], c["Cout"], c["H"], c["W"])
    assert plan.kernel == "tc_bf16_head"
    y, _ = run_chunks(plan, dev["x"], dev["w"], dev["b"], dev.get("r"), c["chunks"][0])
    u1 = run_chunks_u8(plan, dev["x"], dev["w"], dev["b"], dev.get("r"), c["chunks"][0])
    u2 = run_chunks_u8(plan, dev["x"], dev["w"], dev["b"], dev.get("r"), c["chunks"][1])
    assert plan.status() == 0
    assert torch.equal(u1, u2), c
    got = u1.cpu().numpy()
    assert np.array_equal(got, quant_u8(y)), c
    ref = oracle.conv_whole(to_f64(raw["x"], "bf16"), to_f64(raw["w"], "bf16"), to_f64(raw["b"], "bf16"),
                            to_f64(raw["r"], "bf16") if c["residual"] else None)
    delta = ACC_BOUND * float(np.sqrt(np.mean(ref ** 2)))
    lo, hi = oracle.quantize_u8(ref - delta), oracle.quantize_u8(ref + delta)
    assert np.all((lo <= got) & (got <= hi)), (c, int(((lo > got) | (got > hi)).sum()))
    plan.close()
