"""Paged KV cache: append and GQA decode attention, plain definitions.

Sources:
* "How to build your own LLM runtime from scratch (Towards Data Science)",
  section "What it actually builds": paged KV cache, 16 tokens per 4 KiB page
  (16 tokens x 128 dims x 2 bytes = 4096 bytes per page, per KV head, for K
  and for V separately).
* "Build Crude Implementations for Learning", section "Paged KV cache": a
  sequence's blocks are scattered through one pool and found through a table.
* "How To Build Your Own LLM Runtime From Scratch | daily.dev", second
  question: the softmax must be right when the last page is only partly full.

Layouts (shared with the GPU library only as a written format, not as code):

    pool        [P][Hkv][T][D]   fp16, T = 16 tokens per page, D = 128
    page_table  [B][max_pages]   int32, logical block j of sequence b -> page id
    token t of sequence b sits at pool[page_table[b][t // T]][h][t % T][:]

Attention for query head h uses KV head g = h // (Hq / Hkv) (consecutive query
heads share a KV head, as in grouped-query attention), over the L tokens
0..L-1 of its sequence, with no mask beyond L: a decode query sees the whole
context.  The oracle gathers those L rows into a contiguous array and runs a
two-pass softmax (max first, then exp and sum) in float64.
"""

import numpy as np

PAGE_TOKENS = 16


def kv_append_ref(k_pool, v_pool, page_table, k, v, positions):
    """Write k[b][h][:] and v[b][h][:] at token positions[b] of sequence b.

    k_pool/v_pool are modified in place (numpy fp16 arrays [P][Hkv][T][D]).
    """
    k = np.asarray(k)
    v = np.asarray(v)
    for b in range(k.shape[0]):
        t = int(positions[b])
        page = int(page_table[b][t // PAGE_TOKENS])
        slot = t % PAGE_TOKENS
        k_pool[page, :, slot, :] = k[b]
        v_pool[page, :, slot, :] = v[b]


def gather_contiguous(pool, page_table_row, kv_head, length):
    """Rows 0..length-1 of one sequence for one KV head, as a [length][D] array."""
    rows = []
    for t in range(length):
        page = int(page_table_row[t // PAGE_TOKENS])
        rows.append(pool[page, kv_head, t % PAGE_TOKENS, :])
    return np.stack(rows, axis=0)


def attention_contiguous(q, k_c, v_c, scale):
    """softmax(q . K^T * scale) V for one query vector over a contiguous context.

    Two passes: the maximum score, then exponentials, their sum and the
    weighted sum of values.  Returns (out float64 [D], weights float64 [L]).
    """
    q64 = np.asarray(q, dtype=np.float64)
    k64 = np.asarray(k_c, dtype=np.float64)
    v64 = np.asarray(v_c, dtype=np.float64)
    scores = (k64 @ q64) * float(scale)
    m = scores.max()
    e = np.exp(scores - m)
    p = e / e.sum()
    return p @ v64, p


def paged_attention_ref(q, k_pool, v_pool, page_table, context_lens, scale):
    """q: [B][Hq][D]; returns float64 [B][Hq][D]."""
    q = np.asarray(q)
    bsz, hq, d = q.shape
    hkv = k_pool.shape[1]
    group = hq // hkv
    out = np.zeros((bsz, hq, d), dtype=np.float64)
    for b in range(bsz):
        length = int(context_lens[b])
        if length < 1:
            raise ValueError("context length must be >= 1")
        for g in range(hkv):
            k_c = gather_contiguous(k_pool, page_table[b], g, length)
            v_c = gather_contiguous(v_pool, page_table[b], g, length)
            for h in range(g * group, (g + 1) * group):
                out[b, h], _ = attention_contiguous(q[b, h], k_c, v_c, scale)
    return out
