"""Oracle: fp16 -> int8 absmax/127 quantization of K/V rows (test infrastructure only).

Method (genie-ai-runtime release v0.1.0-alpha.12, "Path I series" rows I1-I2:
per-head conversion with scale capture into a separate scales region; Strata
pull request #2698, "What it does": int8 codes with one FP16 scale per 64
values, group absmax / 127):

  for every group of ``gs`` consecutive values x_0..x_{gs-1} (fp16) of one
  (position, kv head) row:
      amax = max_i |x_i|                      (exact in fp32)
      s    = fp16_round_nearest_even(fp32(amax) / fp32(127))
      c_i  = clamp(round_half_even(fp32(x_i) / fp32(s)), -127, 127)
      (s == 0  =>  every c_i = 0)
  dequantized value:  x^_i = c_i * s   (exact in fp64)

The pages give the absmax/127 rule but not its rounding; the reading taken is
the one above (fp32 IEEE division, RNE to fp16 for the scale, half-even for the
code, symmetric clamp so that -128 is never produced).  Inputs must be finite.
"""

import numpy as np

QMAX = 127


def group_scales(x16: np.ndarray, gs: int) -> np.ndarray:
    """fp16 scale per group of ``gs`` values along the last axis.

    ``x16``: fp16 array [..., D] with D % gs == 0.  Returns fp16 [..., D // gs].
    """
    x16 = np.asarray(x16, dtype=np.float16)
    D = x16.shape[-1]
    assert D % gs == 0, "head_dim must be a multiple of the group size"
    g = x16.astype(np.float32).reshape(x16.shape[:-1] + (D // gs, gs))
    amax = np.max(np.abs(g), axis=-1)                 # exact: |fp16| is an fp32
    s32 = amax / np.float32(QMAX)                     # one IEEE fp32 division
    return s32.astype(np.float16)                     # round to nearest even


def quantize_with_scales(x16: np.ndarray, s16: np.ndarray, gs: int) -> np.ndarray:
    """int8 codes of ``x16`` [..., D] given its fp16 group scales [..., D // gs]."""
    x16 = np.asarray(x16, dtype=np.float16)
    s16 = np.asarray(s16, dtype=np.float16)
    D = x16.shape[-1]
    xg = x16.astype(np.float32).reshape(x16.shape[:-1] + (D // gs, gs))
    s32 = s16.astype(np.float32)[..., None]
    with np.errstate(divide="ignore", invalid="ignore"):
        r = xg / s32                                  # IEEE fp32 division
    c = np.rint(r)                                    # round half to even
    c = np.where(s32 == 0, np.float32(0), c)          # all-zero group -> code 0
    c = np.clip(c, -QMAX, QMAX)
    return c.astype(np.int8).reshape(x16.shape)


def quantize(x16: np.ndarray, gs: int):
    """(codes int8 [..., D], scales fp16 [..., D // gs]) for fp16 rows ``x16``."""
    s16 = group_scales(x16, gs)
    return quantize_with_scales(x16, s16, gs), s16


def dequantize(codes: np.ndarray, s16: np.ndarray, gs: int) -> np.ndarray:
    """Exact fp64 values c * s of int8 codes [..., D] with fp16 scales [..., D // gs]."""
    codes = np.asarray(codes)
    D = codes.shape[-1]
    c = codes.astype(np.float64).reshape(codes.shape[:-1] + (D // gs, gs))
    s = np.asarray(s16, dtype=np.float16).astype(np.float64)[..., None]
    return (c * s).reshape(codes.shape)
