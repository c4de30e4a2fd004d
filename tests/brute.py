"""Brute-force restatement of the n-gram hash, for tiny inputs only.

Independent of the C oracle: Python big integers (wrap by ``& (2**64-1)``,
reinterpret as signed by subtracting 2**64), Python's floored ``%``, and each
n-gram built as an explicit tuple straight from the sequence's history of
compressed tokens, with no cache array and no rolling state.

Definition followed ("DeepSeek V4.1", blocks/stack-hashes page, the n-gram hash
``forward``): the n-gram of size n at position p takes the tokens at p, p-1, ...,
p-n+1; slot s (and every later slot) becomes the pad id once a slot at or before
it falls before position 0 or holds a masked (DEAD) token; the slots are
multiplied by the layer's multipliers, XOR-ed, reduced with a floored mod by
the (n-gram size, head) prime and shifted by that column's offset.
"""
from __future__ import annotations

M64 = (1 << 64) - 1


def _signed(v: int) -> int:
    return v - (1 << 64) if v >= (1 << 63) else v


def ngram(history: dict, p: int, n: int, dead: int, pad: int) -> tuple:
    """history: position -> compressed token (missing positions count as DEAD)."""
    out, blocked = [], False
    for s in range(n):
        q = p - s
        if q < 0 or history.get(q, dead) == dead:
            blocked = True
        out.append(pad if blocked else history[q])
    return tuple(out)


def hash_ngram(gram: tuple, mults, prime: int, offset: int) -> int:
    acc = 0
    for tok, m in zip(gram, mults):
        acc ^= (int(tok) * int(m)) & M64
    return _signed(acc) % int(prime) + int(offset)


def compress(raw_id: int, keep: bool, token_map, dead: int) -> int:
    if not keep or raw_id < 0 or raw_id >= len(token_map):
        return dead
    return int(token_map[raw_id])


def hashes_at(history: dict, p: int, lay) -> list:
    """All n_layers x C hash ids of position p, in (layer, column) order."""
    out = []
    N, H = lay.max_ngram, lay.n_heads
    for l in range(lay.n_layers):
        row = []
        for n in range(2, N + 1):
            gram = ngram(history, p, n, lay.dead, lay.pad_id)
            for h in range(H):
                col = (n - 2) * H + h
                row.append(hash_ngram(gram, lay.multipliers[l][:n], lay.primes[l][n - 2][h], lay.offsets[l][col]))
        out.append(row)
    return out
