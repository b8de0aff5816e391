"""fp8 E4M3 KV cache: the comparison format (oracle; test infrastructure only).

Source: the "Quasar" (q27) engine wiki, "KV cache" bullet of the stack list:
the server's default KV format stores K and V as fp8 E4M3 with a scale-free,
saturating conversion (the measured absolute maximum sits well below the
format's 448, so per-row scales buy nothing).  No rotation is applied in that
format; queries and outputs stay in the ordinary basis.

E4M3 (the variant without infinities): 1 sign bit, 4 exponent bits with bias
7, 3 mantissa bits.  Exponent field 0 holds the subnormals m * 2^-9; fields
1..15 hold (8 + m) * 2^(e - 10); the pattern S.1111.111 is NaN, so the largest
finite magnitude is 1.75 * 2^8 = 448.

Reading taken here (the pages name the format and "saturating", nothing
more): a float32 input is rounded to the nearest representable value, ties to
the even mantissa, and magnitudes above 448 become 448 with the input's sign;
a zero result keeps the input's sign (-0 is the byte 0x80).  A non-finite
input is flagged (status bit 1); its byte is NaN (0x7F / 0xFF) for NaN and
+-448 for an infinity.

Record: the 256 code bytes of one head vector, dims in order.  Pool layout as
the 3-bit cache's, with 256-byte records:
offset = ((((page * layers + layer) * kv_heads + head) * 2 + kv) * 256 + row) * 256.

Attention over this cache is the plain formula: s_p = q . k_p / 16 over the
visible positions, P = softmax(s), out = sum_p P_p v_p, in float64 over the
exactly decoded values.
"""
from __future__ import annotations

import numpy as np

RECORD_BYTES = 256
PAGE_SIZE = 256
MAX_FINITE = 448.0
SOFTMAX_SCALE = 1.0 / 16.0


def decode(codes: np.ndarray) -> np.ndarray:
    """E4M3 bytes -> float64 values (NaN for the two NaN patterns)."""
    c = np.asarray(codes, np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    mag = np.where(e == 0, m * 2.0 ** -9, (8 + m) * np.exp2(e - 10.0))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return sign * mag


def _magnitude_code(a: np.ndarray) -> np.ndarray:
    """Nearest E4M3 magnitude code (ties to even) of finite a >= 0, saturating at 448."""
    a = np.asarray(a, np.float64)
    _, E = np.frexp(a)                       # a = f 2^E, f in [0.5, 1): floor(log2 a) = E - 1
    e_unb = np.maximum(E - 1, -6)            # binade; below 2^-6 the subnormal quantum 2^-9
    quantum = np.exp2(e_unb - 3.0)
    r = np.round(a / quantum)                # exact division by a power of two; round half to even
    v = np.minimum(r * quantum, MAX_FINITE)  # the rounded magnitude (may be the next binade's first)
    # encode the rounded value
    _, E2 = np.frexp(np.where(v > 0, v, 1.0))
    e2 = E2 - 1
    normal = v >= 2.0 ** -6
    exp_field = np.where(normal, e2 + 7, 0)
    mant = np.where(normal, v / np.exp2(e2 - 3.0) - 8, v / 2.0 ** -9)
    return (exp_field.astype(np.int64) << 3) | mant.astype(np.int64)


def encode(x: np.ndarray):
    """float32 (or bf16-exact) inputs -> (E4M3 bytes uint8, non-finite flags int32), elementwise."""
    x = np.asarray(x, np.float32).astype(np.float64)
    finite = np.isfinite(x)
    a = np.where(finite, np.abs(x), 0.0)
    code = _magnitude_code(a)
    code = np.where(np.isinf(x), 0x7E, code)
    code = np.where(np.isnan(x), 0x7F, code)
    sign = np.signbit(x) & ~np.isnan(x)
    code = code | np.where(sign, 0x80, 0)
    return code.astype(np.uint8), (~finite).astype(np.int32)


def encode_vectors(x_raw: np.ndarray):
    """Raw head vectors [..., 256] -> (records uint8 [..., 256], flag per vector)."""
    codes, nf = encode(x_raw)
    return codes, nf.reshape(nf.shape[:-1] + (-1,)).max(axis=-1)


def attention(q: np.ndarray, k_hat: np.ndarray, v_hat: np.ndarray, n_ctx: int, group: int) -> np.ndarray:
    """Verify attention of one slot in the plain basis, float64.

    q [T, Hq, D]; k_hat, v_hat [Hkv, L, D] decoded values; query token t sees
    positions [0, n_ctx + t]; q head h reads kv head h // group.
    """
    q = np.asarray(q, np.float64)
    T, Hq, D = q.shape
    out = np.zeros((T, Hq, D), np.float64)
    for h in range(Hq):
        g = h // group
        for t in range(T):
            lim = n_ctx + t + 1
            s = (np.asarray(k_hat[g, :lim], np.float64) @ q[t, h]) * SOFTMAX_SCALE
            e = np.exp(s - np.max(s))
            out[t, h] = (e @ np.asarray(v_hat[g, :lim], np.float64)) / np.sum(e)
    return out


class Fp8PagedCache:
    """A slot's position p lives in page page_table[p // 256], row p % 256 (as the 3-bit cache)."""

    def __init__(self, num_pages: int, num_layers: int, num_kv_heads: int):
        self.num_pages = num_pages
        self.num_layers = num_layers
        self.num_kv_heads = num_kv_heads
        self.pool = np.zeros(num_pages * num_layers * num_kv_heads * 2 * PAGE_SIZE * RECORD_BYTES, np.uint8)

    def _offsets(self, page_table_row, positions, layer, kv_head, kv):
        positions = np.asarray(positions, np.int64)
        pages = np.asarray(page_table_row, np.int64)[positions // PAGE_SIZE]
        if np.any(pages < 0) or np.any(pages >= self.num_pages):
            raise IndexError("page id out of range")
        L, H = self.num_layers, self.num_kv_heads
        return ((((pages * L + layer) * H + kv_head) * 2 + kv) * PAGE_SIZE + positions % PAGE_SIZE) * RECORD_BYTES

    def append(self, page_table_row, start: int, layer: int, k_raw: np.ndarray, v_raw: np.ndarray) -> np.ndarray:
        """Encode raw K, V [n, Hkv, 256] at positions [start, start + n); returns flags [n, Hkv, 2]."""
        n = k_raw.shape[0]
        flags = np.zeros((n, self.num_kv_heads, 2), np.int32)
        pos = np.arange(start, start + n)
        for kv, x in ((0, k_raw), (1, v_raw)):
            for g in range(self.num_kv_heads):
                rec, f = encode_vectors(x[:, g, :])
                off = self._offsets(page_table_row, pos, layer, g, kv)
                self.pool[off[:, None] + np.arange(RECORD_BYTES)[None, :]] = rec
                flags[:, g, kv] = f
        return flags

    def records(self, page_table_row, layer: int, kv_head: int, kv: int, start: int, count: int) -> np.ndarray:
        off = self._offsets(page_table_row, np.arange(start, start + count), layer, kv_head, kv)
        return self.pool[off[:, None] + np.arange(RECORD_BYTES)[None, :]]

    def decoded(self, page_table_row, layer: int, kv_head: int, kv: int, count: int) -> np.ndarray:
        return decode(self.records(page_table_row, layer, kv_head, kv, 0, count))

    def verify(self, page_table_row, layer: int, n_ctx: int, q: np.ndarray, group: int) -> np.ndarray:
        L = n_ctx + q.shape[0]
        kh = np.stack([self.decoded(page_table_row, layer, g, 0, L) for g in range(self.num_kv_heads)])
        vh = np.stack([self.decoded(page_table_row, layer, g, 1, L) for g in range(self.num_kv_heads)])
        return attention(q, kh, vh, n_ctx, group)
