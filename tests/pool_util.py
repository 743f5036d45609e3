"""Synthetic paged indexer pools for tests (host side, numpy)."""
import numpy as np

import oracle

PAGE = 128


def make_pool(B, max_tokens, seed, num_kv_heads=2, pool_head_dim=384, head_size=256, spare_pages=3,
              unused_slots=()):
    """Every sequence gets ceil(max_tokens/128) K pages and as many V pages, drawn as a random
    permutation of the pool's pages (V ids offset by +numPages); `unused_slots` lists
    (b, plane, slot) entries set to -1.  The pool starts filled with a sentinel."""
    rng = np.random.default_rng(seed)
    per_seq = (max_tokens + PAGE - 1) // PAGE
    num_pages = B * per_seq + spare_pages
    k_ids = rng.permutation(num_pages)[:B * per_seq].reshape(B, per_seq)
    v_ids = rng.permutation(num_pages)[:B * per_seq].reshape(B, per_seq) + num_pages
    max_pages = per_seq + 1                      # one spare slot per sequence, left unused
    table = np.full((B, 2, max_pages), -1, np.int32)
    table[:, 0, :per_seq] = k_ids
    table[:, 1, :per_seq] = v_ids
    for b, plane, slot in unused_slots:
        table[b, plane, slot] = -1
    pool = np.full((2 * num_pages, PAGE, num_kv_heads, pool_head_dim), 0x5A5A, np.uint16)
    return oracle.Pool(pool, table, num_pages, num_kv_heads, pool_head_dim, head_size)


def k_tail(pool, b, t):
    page = pool.page_table[b, 0, t // PAGE]
    return None if page < 0 else pool.pool[page, t % PAGE, 0, pool.head_size:pool.head_size + 128]


def v_tail(pool, b, g):
    page = pool.page_table[b, 1, (4 * g) // PAGE]
    return None if page < 0 else pool.pool[page, (4 * g) % PAGE, 0, pool.head_size:pool.head_size + 128]
