"""Oracle of the batched packed-cache row operations.

TEST INFRASTRUCTURE ONLY, like the rest of this package: the CUDA library
never imports it.

What it follows: page "@mlx-bun/inference 0.0.0-stage -> 1.0.0", files
package/src/model/batched-quant.ts (mergeQuantRows, extendQuantRows,
extractQuantRow, filterQuantRows) and package/src/model/batched-mask.ts
(mergeKVRows, extendKVRows, extractKVRow): continuous batching moves whole
token rows of a quantized cache between batch rows. Quantization packs along
head_dim only, so every token is a whole row of each packed buffer and these
operations copy bytes without touching a quantization group. Rows are
right-justified: a row shorter than the batch width is padded on the LEFT
with zero bytes, and the per-row pad counts travel with the batch.

A cache here is the dict of five numpy arrays the codec oracle uses
(k_codes, k_scales, k_zeros, v_codes, v_scales), each [B, H, S, X]; S is the
number of valid token columns (the window), as in the pages' offset-trimmed
arrays. The definitions below are the pages' operations written out with
numpy zeros, concatenation, slicing and take; nothing here is tuned.
"""
from __future__ import annotations

import numpy as np

BUFFERS = ("k_codes", "k_scales", "k_zeros", "v_codes", "v_scales")


def _left_pad(a: np.ndarray, pad: int) -> np.ndarray:
    """Zero tokens in front of axis 2 (leftPadTo)."""
    if pad == 0:
        return a.copy()
    B, H, _, X = a.shape
    return np.concatenate([np.zeros((B, H, pad, X), a.dtype), a], axis=2)


def merge_rows(rows: list) -> tuple:
    """mergeQuantRows: stack single-row caches ([1, H, L_i, X] each) into one
    left-padded [N, H, W, X] batch, W = max L_i, pad_i = W - L_i."""
    lens = [r["k_codes"].shape[2] for r in rows]
    width = max(lens)
    pads = [width - n for n in lens]
    out = {name: np.concatenate([_left_pad(r[name], p) for r, p in zip(rows, pads)], axis=0) for name in BUFFERS}
    return out, pads, width


def extend_rows(batch: dict, pads: list, row: dict) -> tuple:
    """extendQuantRows: append one right-justified row to a batch; whichever
    side is narrower is padded on the left to the common width; existing
    pads grow by the batch side's pad, never shrink."""
    S = batch["k_codes"].shape[2]
    Lr = row["k_codes"].shape[2]
    width = max(S, Lr)
    out = {name: np.concatenate([_left_pad(batch[name], width - S), _left_pad(row[name], width - Lr)], axis=0)
           for name in BUFFERS}
    return out, [p + (width - S) for p in pads] + [width - Lr], width


def extract_row(batch: dict, pad: int, i: int) -> dict:
    """extractQuantRow: batch row i past its left pad, as a contiguous
    single-row cache [1, H, S - pad, X]."""
    S = batch["k_codes"].shape[2]
    return {name: np.ascontiguousarray(batch[name][i:i + 1, :, pad:S]) for name in BUFFERS}


def filter_rows(batch: dict, keep: list) -> dict:
    """filterQuantRows: keep the batch rows `keep` (in that order)."""
    idx = np.asarray(keep, dtype=np.int64)
    return {name: np.take(batch[name], idx, axis=0) for name in BUFFERS}
