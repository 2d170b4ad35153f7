"""Test helper: a DCP rank's compact pool built from a global paged cache.

Partition r's owned rows (global tokens t = r + jP) are copied, in local order
j, into pages drawn at random from a rank pool; req_to_token[b][j] is the
slot (64 page + row) of local token j.  Pure data movement: no attention
arithmetic lives here.
"""
import numpy as np


def compact_pool(kv_bits, block_table, seq_lens, part_id, num_parts, rng, spare_pages=3,
                 page_size=64, extra_slots=64):
    kv_bits = np.asarray(kv_bits)
    B = len(seq_lens)
    local = [int(L) // num_parts + int(part_id < int(L) % num_parts) for L in seq_lens]
    need = [-(-n // page_size) for n in local]
    pool = sum(need) + spare_pages
    perm = rng.permutation(pool)
    width = max(1, max(need)) * page_size + extra_slots
    pool_bits = np.zeros((pool,) + kv_bits.shape[1:], dtype=kv_bits.dtype)
    r2t = np.full((B, width), -7, dtype=np.int32)       # slots past a request: never read
    pages = []
    off = 0
    for b in range(B):
        mine = perm[off:off + need[b]]
        off += need[b]
        pages.append([int(p) for p in mine])
        for j in range(local[b]):
            t = part_id + j * num_parts
            g_page, g_row = int(block_table[b][t // page_size]), t % page_size
            l_page, l_row = int(mine[j // page_size]), j % page_size
            pool_bits[l_page, l_row] = kv_bits[g_page, g_row]
            r2t[b, j] = l_page * page_size + l_row
    return pool_bits, r2t, pages, local
