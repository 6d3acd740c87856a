"""Oracle for DynamicQuant of q^N (per-row symmetric int8 quantisation).

Test infrastructure only (see oracle/__init__.py). Written from the page
"aclnnMlaPrologV3WeightNz" ("Formula", Dequant Scale Query Nope):
dequantScaleQNope = RowMax(abs(q^N)) / 127 and q^N = round(q^N /
dequantScaleQNope), with the scale of shape (T, N, 1) ("Shape restrictions"),
i.e. one scale per token and head, the row being the last axis (Hckv).

Readings where the page is silent:
* round is round-half-to-even (the pages state their formulas in PyTorch
  terms; torch.round ties to even); codes are clamped to [-127, 127];
* the code is an integer decided by floating point, so it is decided in
  float32 (the precision of the GPU path): scale = fl32(rowmax / 127),
  v = fl32(q / scale), code = rint(v). RowMax is exact in any precision, and
  16-bit inputs widen to float32 exactly;
* an all-zero row has scale 0 and codes 0 (the formula would divide 0 by 0).
"""
import numpy as np


def ref_dynamic_quant(q):
    """q: float64 [rows, H] holding 16-bit input values. Returns
    (codes int8 [rows, H], scale float32 [rows])."""
    q32 = np.asarray(q, dtype=np.float64).astype(np.float32)
    rowmax = np.max(np.abs(q32), axis=-1)
    scale = (rowmax / np.float32(127.0)).astype(np.float32)
    safe = np.where(scale > 0, scale, np.float32(1.0)).astype(np.float32)
    v = (q32 / safe[:, None]).astype(np.float32)
    codes = np.clip(np.rint(v), -127, 127)
    codes[scale == 0] = 0
    return codes.astype(np.int8), scale
