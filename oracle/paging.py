"""Paged cache addressing with a 256-raw-position logical block (oracle; test infrastructure only).

[P2] "DeepSeek V4 稀疏注意力完全解剖", 设计 1：统一的"逻辑 block size": whatever the
cache kind, one block covers 256 raw token positions, so a c4a block holds
256/4 = 64 compressed entries, a c128a block 256/128 = 2, an SWA block 256 raw
tokens.  [P1] §2.2 (PagedAttention): per-request block tables map logical blocks
to physical blocks that need not be contiguous.

Reading: compressed entry i of a kind with stride s starts at raw position s*i, so it
is placed in logical block floor(i / (256/s)), slot i mod (256/s).
"""
import numpy as np

LOGICAL_BLOCK_POSITIONS = 256


class PagingError(ValueError):
    """A row was needed from a logical block that the table does not map."""


def entries_per_block(stride):
    """Rows per block for a cache kind whose entries advance ``stride`` raw positions."""
    assert LOGICAL_BLOCK_POSITIONS % stride == 0
    return LOGICAL_BLOCK_POSITIONS // stride


def physical_rows(table_row, logical_ids, epb, num_blocks):
    """Physical row ids (block * epb + slot) of logical rows, via one request's table.

    Raises PagingError when a needed block is unmapped (id < 0), out of the pool, or
    beyond the table.
    """
    ids = np.asarray(logical_ids, dtype=np.int64)
    blk_idx = ids // epb
    if np.any(ids < 0) or np.any(blk_idx >= len(table_row)):
        raise PagingError("logical row beyond the block table")
    blk = np.asarray(table_row, dtype=np.int64)[blk_idx]
    if np.any(blk < 0) or np.any(blk >= num_blocks):
        raise PagingError("logical row in an unmapped block")
    return blk * epb + ids % epb


def gather(pool_rows, table_row, logical_ids, epb):
    """Rows of a pool viewed as [num_blocks * epb, ...] for the given logical ids."""
    num_blocks = pool_rows.shape[0] // epb
    return pool_rows[physical_rows(table_row, logical_ids, epb, num_blocks)]


def scatter(pool_rows, table_row, logical_ids, epb, values):
    """Write rows into a pool viewed as [num_blocks * epb, ...] (in place)."""
    num_blocks = pool_rows.shape[0] // epb
    pool_rows[physical_rows(table_row, logical_ids, epb, num_blocks)] = values
