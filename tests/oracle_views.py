"""Test-side views of the oracle on parts of a large weight.

The oracle's steps are per block (codes), per group (double quant) and per
weight (dequant), so the dequantized rows or columns of a big weight follow
from the absmax of every block plus the codes of the blocks asked for. This
module only selects blocks; all arithmetic is the oracle's.
"""
import numpy as np

from oracle import nf4_oracle as o


class OracleWeight:
    """dtype "nf4" / "fp4": codes per block, double quant over all blocks;
    "int8": every block on its own (its absmax is its scale)."""

    def __init__(self, W: np.ndarray, dtype: str = "nf4"):
        self.W = np.ascontiguousarray(W, dtype=np.float32)
        self.dtype = dtype
        self.N, self.K = self.W.shape
        self.nblk = self.K // o.BLOCKSIZE
        if dtype != "int8":
            self.levels = o.levels_of(dtype)
            self.absmax = o.block_absmax(self.W.reshape(-1))
            self.a8, self.s2 = o.double_quant(self.absmax)
            self.ahat = o.dequant_absmax(self.a8, self.s2)

    def _blocks(self, block_ids: np.ndarray) -> np.ndarray:
        wb = self.W.reshape(-1, o.BLOCKSIZE)[block_ids]
        if self.dtype == "int8":
            q, a = o.int8_quantize_flat(wb.reshape(-1))
            return o.int8_dequantize_flat(q, a).reshape(-1, o.BLOCKSIZE)
        codes = o.quantize_codes(wb.reshape(-1), self.absmax[block_ids], self.levels)
        return o.dequantize_codes(codes.reshape(-1, o.BLOCKSIZE), self.ahat[block_ids],
                                  self.levels)

    def rows(self, rows) -> np.ndarray:
        rows = np.asarray(rows, dtype=np.int64)
        ids = (rows[:, None] * self.nblk + np.arange(self.nblk)[None, :]).reshape(-1)
        return self._blocks(ids).reshape(rows.size, self.K)

    def col_blocks(self, kblocks) -> np.ndarray:
        """Dequantized columns of the given 64-column blocks: [N, 64 * len]."""
        kb = np.asarray(kblocks, dtype=np.int64)
        ids = (np.arange(self.N)[:, None] * self.nblk + kb[None, :]).reshape(-1)
        return self._blocks(ids).reshape(self.N, kb.size * o.BLOCKSIZE)

    @staticmethod
    def columns_of(kblocks) -> np.ndarray:
        kb = np.asarray(kblocks, dtype=np.int64)
        return (kb[:, None] * o.BLOCKSIZE + np.arange(o.BLOCKSIZE)[None, :]).reshape(-1)


def sample_indices(n: int, count: int, seed: int) -> np.ndarray:
    """Sorted sample of `count` indices of range(n), always holding 0 and n-1."""
    rng = np.random.default_rng(seed)
    pick = set([0, n - 1])
    if count >= n:
        return np.arange(n)
    while len(pick) < count:
        pick.add(int(rng.integers(0, n)))
    return np.array(sorted(pick), dtype=np.int64)
