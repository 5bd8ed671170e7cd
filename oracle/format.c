/*
 * CPU oracle: the cache record format, written from its specification.
 *
 * TEST INFRASTRUCTURE ONLY (see affine.c).  The CUDA library implements the
 * same format independently; this file is the plain statement the tests
 * compare its bytes against.
 *
 * The pages fix only that every token's record has a fixed size, so its
 * address follows from the token index alone ("D-Quant", Sec. 4.2 Eq. (3)
 * and App. A after Eq. (9)).  The bit layout inside a record is this
 * library's own choice, specified here:
 *
 * A record is an array of little-endian 32-bit words.  With b in {2, 4}
 * bits per code, each 16-bit half of a word holds F = 16/b fields; field f
 * occupies bits [b*f, b*f + b) of its half.  With b = 3 the record is a
 * 2-bit plane (the low two bits of every code, laid out as b = 2) followed
 * by a 1-bit plane (bit 2 of every code, F = 16) whose field f sits at bit
 * P(f) of its half, P(f) = 2f + 2 for f <= 6, 0 for f = 7, 2f - 13 for
 * 8 <= f <= 14 and 1 for f = 15 (a permutation of 0..15: the bits of the
 * fields that a reader turns into operands together then need few distinct
 * shifts to meet their 2-bit fields).
 *
 * Key row of token t (d channels, one record per token):
 *   channel c -> e = c & 1, tig = (c >> 1) & 3, sub = (c >> 3) & 1, i = c >> 4
 *   r = 2*i + sub, idx = tig*(d/8) + r
 *   word = idx / F, half = e, field = idx % F
 * Value pair record of tokens (2p, 2p+1) (one record per token pair):
 *   channel c -> g = c & 7, h = (c >> 3) & 1, mi = c >> 4
 *   r = 2*mi + h, idx = g*(d/8) + r
 *   word = idx / F, half = t & 1, field = idx % F
 */
#include <stdint.h>
#include <string.h>

static int fields_per_half(int b) { return 16 / b; }

/* Bit position of (channel c, half e) in a record laid out for b in {2, 4}. */
static long bitpos(int idx, int e, int b) {
    int F = fields_per_half(b);
    return 32L * (idx / F) + 16L * e + (long)b * (idx % F);
}

/* Bit position of field idx, half e, in the 1-bit plane of a 3-bit record. */
static long bitpos1(int idx, int e) {
    int f = idx % 16;
    int p = f <= 6 ? 2 * f + 2 : (f == 7 ? 0 : (f == 15 ? 1 : 2 * f - 13));
    return 32L * (idx / 16) + 16L * e + p;
}

static int k_idx(int c, int d) {
    int tig = (c >> 1) & 3, sub = (c >> 3) & 1, i = c >> 4;
    return tig * (d / 8) + 2 * i + sub;
}

static int v_idx(int c, int d) {
    int g = c & 7, h = (c >> 3) & 1, mi = c >> 4;
    return g * (d / 8) + 2 * mi + h;
}

static void put_bits(uint8_t *rec, long pos, int b, unsigned v) {
    for (int k = 0; k < b; k++) {
        long p = pos + k;
        if ((v >> k) & 1u) rec[p >> 3] |= (uint8_t)(1u << (p & 7));
        else rec[p >> 3] &= (uint8_t)~(1u << (p & 7));
    }
}

static unsigned get_bits(const uint8_t *rec, long pos, int b) {
    unsigned v = 0;
    for (int k = 0; k < b; k++) {
        long p = pos + k;
        v |= (unsigned)((rec[p >> 3] >> (p & 7)) & 1u) << k;
    }
    return v;
}

/* Bytes in one key row / one value pair record. */
int or_k_row_bytes(int d, int b) { return d * b / 8; }
int or_v_pair_bytes(int d, int b) { return 2 * d * b / 8; }

/* Key row: write codes[d] of one token. */
void or_pack_k_row(const unsigned char *codes, int d, int b, uint8_t *row) {
    memset(row, 0, (size_t)or_k_row_bytes(d, b));
    for (int c = 0; c < d; c++) {
        int idx = k_idx(c, d), e = c & 1;
        if (b == 3) {
            put_bits(row, bitpos(idx, e, 2), 2, codes[c] & 3u);
            put_bits(row + d / 4, bitpos1(idx, e), 1, (codes[c] >> 2) & 1u);
        } else {
            put_bits(row, bitpos(idx, e, b), b, codes[c]);
        }
    }
}

void or_unpack_k_row(const uint8_t *row, int d, int b, unsigned char *codes) {
    for (int c = 0; c < d; c++) {
        int idx = k_idx(c, d), e = c & 1;
        if (b == 3)
            codes[c] = (unsigned char)(get_bits(row, bitpos(idx, e, 2), 2) |
                                       (get_bits(row + d / 4, bitpos1(idx, e), 1) << 2));
        else
            codes[c] = (unsigned char)get_bits(row, bitpos(idx, e, b), b);
    }
}

/* Value pair record: write codes[d] of the token with parity e (0 or 1)
 * into the record of its pair, leaving the other token's bits unchanged. */
void or_pack_v_token(const unsigned char *codes, int d, int b, int e, uint8_t *rec) {
    for (int c = 0; c < d; c++) {
        int idx = v_idx(c, d);
        if (b == 3) {
            put_bits(rec, bitpos(idx, e, 2), 2, codes[c] & 3u);
            put_bits(rec + d / 2, bitpos1(idx, e), 1, (codes[c] >> 2) & 1u);
        } else {
            put_bits(rec, bitpos(idx, e, b), b, codes[c]);
        }
    }
}

void or_unpack_v_token(const uint8_t *rec, int d, int b, int e, unsigned char *codes) {
    for (int c = 0; c < d; c++) {
        int idx = v_idx(c, d);
        if (b == 3)
            codes[c] = (unsigned char)(get_bits(rec, bitpos(idx, e, 2), 2) |
                                       (get_bits(rec + d / 2, bitpos1(idx, e), 1) << 2));
        else
            codes[c] = (unsigned char)get_bits(rec, bitpos(idx, e, b), b);
    }
}

/*
 * Raw (16-bit) region of a unit: slots [0, n_sink) hold the sink tokens,
 * slots n_sink + (t mod n_recent) the recent ring.  Keys are row-major
 * [slot][d]; values are pair-interleaved: element (slot, c) at
 * ((slot >> 1)*d + c)*2 + (slot & 1).
 */
long or_raw_v_index(int slot, int c, int d) {
    return ((long)(slot >> 1) * d + c) * 2 + (slot & 1);
}

int or_raw_slot(long t, int n_sink, int n_recent) {
    if (t < n_sink) return (int)t;
    return n_sink + (int)(t % n_recent);
}
