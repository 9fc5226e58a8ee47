"""Algorithm 1, the block-wise outer loop (exact integer / bf16 bit copies).

TEST INFRASTRUCTURE ONLY (see oracle/__init__.py).

Source: "Nemotron-Labs-TwoTower" wiki, section "Block-wise generation": the context
tower runs once over the prompt; each new block of S positions starts as [MASK] tokens
and is refined by the denoiser (the single-block sampler); once the block is clean it
is committed, the context tower processes the committed tokens causally to update its
caches, and the loop continues with the next block.  The MLX port's README
("Configuration (diffusion)") adds the two stopping knobs: a number of new tokens (a
multiple of the block size) and an end-of-sequence id.

Readings where the pages are silent:
* the context tower's forward needs trained weights; the keys/values it would append
  for a committed block are stood in for by that block's own keys/values (k_blk,
  v_blk), written at logical positions ctx_len .. ctx_len + S - 1 of the sequence's
  cache (rows of a contiguous cache, or rows of the pages the page table names), after
  which ctx_len grows by S;
* a sequence is done after the block in which it commits the end-of-sequence id or in
  which its generated count reaches max_new_tokens; later blocks leave it untouched:
  its block positions hold the pad id, nothing is appended and ctx_len stays;
* the block index of the k-th block of a call is first_block + k (it enters the
  logits stand-in's hash).
"""
import numpy as np


def append_block(cache: dict, k_blk, v_blk, ctx_len, ids, eos_id: int, max_new: int,
                 generated, done) -> dict:
    """One append, every sequence of the batch.

    cache: {"k_ctx", "v_ctx"} bf16 bits [B][Lcap][Hkv][D] (contiguous) or {"k_pages",
    "v_pages", "page_table"} ([P][64][Hkv][D], int [B][max_pages]).  k_blk, v_blk bf16
    bits [B][S][Hkv][D]; ids int [B][S] (the committed block).  Returns a dict with new
    copies of the cache arrays, ctx_len, generated and done.
    """
    out = {k: np.array(v, copy=True) for k, v in cache.items()}
    ctx_len = np.array(ctx_len, np.int64, copy=True)
    generated = np.array(generated, np.int64, copy=True)
    done = np.array(done, np.uint8, copy=True)
    B, S = np.asarray(ids).shape
    for b in range(B):
        if done[b]:
            continue
        for s in range(S):
            pos = int(ctx_len[b]) + s
            if "page_table" in out:
                pg = int(out["page_table"][b, pos // 64])
                out["k_pages"][pg, pos % 64] = k_blk[b, s]
                out["v_pages"][pg, pos % 64] = v_blk[b, s]
            else:
                out["k_ctx"][b, pos] = k_blk[b, s]
                out["v_ctx"][b, pos] = v_blk[b, s]
        ctx_len[b] += S
        generated[b] += S
        if np.any(np.asarray(ids)[b] == eos_id) or generated[b] >= max_new:
            done[b] = 1
    out.update(ctx_len=ctx_len, generated=generated, done=done)
    return out


def generate(B: int, S: int, T: int, mask_id: int, gamma: float, n_blocks: int,
             logits_fn, eos_id: int, pad_id: int, max_new: int, first_block: int = 0) -> dict:
    """Token side of the outer loop: logits_fn(b, block, step, positions) -> [len][V].

    Returns tokens int [B][n_blocks * S] (pad where a sequence was already done), the
    number of steps of every (sequence, block), generated and done.
    """
    from .loop import denoise_block
    tokens = np.full((B, n_blocks * S), pad_id, np.int64)
    steps = np.zeros((B, n_blocks), np.int64)
    generated = np.zeros(B, np.int64)
    done = np.zeros(B, np.uint8)
    for k in range(n_blocks):
        blk = first_block + k
        for b in range(B):
            if done[b]:
                continue
            r = denoise_block(S, T, mask_id, gamma, lambda st, pos, b=b: logits_fn(b, blk, st, pos))
            tokens[b, k * S:(k + 1) * S] = r["ids"]
            steps[b, k] = r["steps"]
            generated[b] += S
            if np.any(r["ids"] == eos_id) or generated[b] >= max_new:
                done[b] = 1
    return dict(tokens=tokens, steps=steps, generated=generated, done=done)
