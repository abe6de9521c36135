/*
 * SplitZip BF16 codec -- CPU ORACLE (test infrastructure only; see sz_oracle.h).
 *
 * Plain loops, one element at a time, in the order the pages describe the
 * method ([P1] "splitzip_codec.py": calibrate_codebook, _align4,
 * assemble_payload, encode_torch, decode_torch).  Nothing here is blocked,
 * fused, vectorised or reordered.
 */
#include "sz_oracle.h"

#include <string.h>

/* [P1] _align4: round a byte offset up to a multiple of 4. */
static uint64_t align4(uint64_t v) { return (v + 3u) & ~(uint64_t)3u; }

/* [P1] module docstring: the exponent is bits 7..14 of the pattern. */
static uint8_t exponent_byte(uint16_t x) { return (uint8_t)((x >> 7) & 0xFFu); }

/* [P1] module docstring / encode_torch: the sign bit (bit 15) goes to bit 7
 * of the sm byte, the low 7 mantissa bits stay in bits 0..6. */
static uint8_t sign_mantissa_byte(uint16_t x) {
  return (uint8_t)(((x >> 8) & 0x80u) | (x & 0x7Fu));
}

/* [P1] module docstring: the sign goes back to bit 15, the exponent to bits
 * 7..14, the low mantissa stays in bits 0..6 (the reconstruction merge). */
static uint16_t merge(uint8_t sm, uint8_t exp) {
  return (uint16_t)(((uint32_t)(sm & 0x80u) << 8) | ((uint32_t)exp << 7) | (uint32_t)(sm & 0x7Fu));
}

void szo_histogram(const uint16_t* x, uint64_t n, uint64_t hist[256]) {
  for (int v = 0; v < 256; ++v) hist[v] = 0;
  for (uint64_t i = 0; i < n; ++i) hist[exponent_byte(x[i])] += 1;
}

void szo_select(const uint64_t hist[256], uint64_t n, szo_codebook* cb) {
  /* Order the 256 exponent values by count, largest first.  The insertion
   * sort below is stable over the ascending value order it starts from, so
   * equal counts keep ascending value order (the tie rule of this codec). */
  int order[256];
  for (int v = 0; v < 256; ++v) order[v] = v;
  for (int i = 1; i < 256; ++i) {
    int v = order[i];
    int j = i - 1;
    while (j >= 0 && hist[order[j]] < hist[v]) {
      order[j + 1] = order[j];
      --j;
    }
    order[j + 1] = v;
  }

  /* [P1] calibrate_codebook: top = min(16, number of distinct values). */
  uint32_t distinct = 0;
  for (int v = 0; v < 256; ++v) distinct += (hist[v] > 0) ? 1u : 0u;
  uint32_t top = distinct < 16u ? distinct : 16u;

  for (int v = 0; v < 256; ++v) cb->enc_lut[v] = (uint8_t)SZO_ESCAPE;
  for (int c = 0; c < 16; ++c) cb->dec_lut[c] = 0;
  uint64_t top_count = 0;
  for (uint32_t code = 0; code < top; ++code) {
    int value = order[code];
    cb->enc_lut[value] = (uint8_t)code;
    cb->dec_lut[code] = (uint8_t)value;
    top_count += hist[value];
  }
  cb->n_top = top;
  cb->top_count = top_count;
  /* [P1] coverage = sum of top counts / sum of all counts (= n). */
  cb->coverage = (n == 0) ? 1.0 : (double)top_count / (double)n;
}

void szo_calibrate(const uint16_t* x, uint64_t n, szo_codebook* cb) {
  uint64_t hist[256];
  szo_histogram(x, n, hist);
  szo_select(hist, n, cb);
}

void szo_layout(uint64_t n, uint64_t n_esc, double coverage, szo_meta* m) {
  /* [P1] assemble_payload, offsets in stream order. */
  m->n = n;
  m->n_pairs = (n + 1) / 2;
  m->n_esc = n_esc;
  m->chunk_size = SZO_CHUNK;
  m->off_pk = 0;
  m->off_sm = align4(m->off_pk + m->n_pairs);
  m->off_cid = align4(m->off_sm + n);
  m->off_lpos = m->off_cid + 4 * n_esc;
  m->off_ev = align4(m->off_lpos + 2 * n_esc);
  m->comp_bytes = m->off_ev + n_esc;
  m->coverage = coverage;
}

uint64_t szo_count_escapes(const uint16_t* x, uint64_t n, const szo_codebook* cb) {
  uint64_t e = 0;
  for (uint64_t i = 0; i < n; ++i)
    if (cb->enc_lut[exponent_byte(x[i])] == SZO_ESCAPE) e += 1;
  return e;
}

static void put_le32(uint8_t* p, uint32_t v) {
  p[0] = (uint8_t)(v & 0xFFu);
  p[1] = (uint8_t)((v >> 8) & 0xFFu);
  p[2] = (uint8_t)((v >> 16) & 0xFFu);
  p[3] = (uint8_t)((v >> 24) & 0xFFu);
}

static void put_le16(uint8_t* p, uint32_t v) {
  p[0] = (uint8_t)(v & 0xFFu);
  p[1] = (uint8_t)((v >> 8) & 0xFFu);
}

static uint32_t get_le32(const uint8_t* p) {
  return (uint32_t)p[0] | ((uint32_t)p[1] << 8) | ((uint32_t)p[2] << 16) | ((uint32_t)p[3] << 24);
}

static uint32_t get_le16(const uint8_t* p) { return (uint32_t)p[0] | ((uint32_t)p[1] << 8); }

int szo_encode(const uint16_t* x, uint64_t n, const szo_codebook* cb,
               uint8_t* out, uint64_t capacity, szo_meta* m) {
  /* The escape count fixes the positions of the last two sections, so it is
   * counted first ([P1] encode_torch gets it from nonzero() before
   * assemble_payload places the streams). */
  uint64_t n_esc = szo_count_escapes(x, n, cb);
  szo_layout(n, n_esc, cb->coverage, m);
  if (m->comp_bytes > capacity) return SZO_ERR_CAPACITY;

  /* [P1] assemble_payload starts from a zero-filled buffer: every pad byte
   * and the pad nibble of an odd n stay 0. */
  memset(out, 0, m->comp_bytes);

  uint64_t k = 0; /* escapes listed so far, in ascending element index */
  for (uint64_t i = 0; i < n; ++i) {
    uint8_t exp = exponent_byte(x[i]);
    uint8_t code = cb->enc_lut[exp];            /* [P1] enc_lut_marked[exp]  */
    uint8_t nibble = (uint8_t)(code & 0x0Fu);   /* escape mark 16 -> code 0  */
    /* element 2j -> low nibble of pk[j], element 2j+1 -> high nibble */
    out[m->off_pk + i / 2] |= (uint8_t)(nibble << (4 * (i % 2)));
    out[m->off_sm + i] = sign_mantissa_byte(x[i]);
    if (code == SZO_ESCAPE) {
      /* [P1] encode_torch: chunk_id = idx // chunk, local_pos = idx % chunk
       * (uint16 little-endian), esc_val = the raw exponent byte. */
      put_le32(out + m->off_cid + 4 * k, (uint32_t)(i / SZO_CHUNK));
      put_le16(out + m->off_lpos + 2 * k, (uint32_t)(i % SZO_CHUNK));
      out[m->off_ev + k] = exp;
      k += 1;
    }
  }
  return SZO_OK;
}

int szo_decode(const uint8_t* payload, const szo_meta* m, const uint8_t dec_lut[16], uint16_t* out) {
  szo_meta expect;
  szo_layout(m->n, m->n_esc, m->coverage, &expect);
  if (m->chunk_size != SZO_CHUNK || m->n_esc > m->n || m->n_pairs != expect.n_pairs ||
      m->off_pk != expect.off_pk || m->off_sm != expect.off_sm || m->off_cid != expect.off_cid ||
      m->off_lpos != expect.off_lpos || m->off_ev != expect.off_ev ||
      m->comp_bytes != expect.comp_bytes)
    return SZO_ERR_META;

  /* [P1] decode_torch, dense part: code of element i from its nibble, the
   * exponent from dec_lut, then the bitwise merge with the sm byte. */
  for (uint64_t i = 0; i < m->n; ++i) {
    uint8_t byte = payload[m->off_pk + i / 2];
    uint8_t code = (uint8_t)((byte >> (4 * (i % 2))) & 0x0Fu);
    uint8_t exp = dec_lut[code];
    out[i] = merge(payload[m->off_sm + i], exp);
  }
  /* [P1] decode_torch, escape part: idx = chunk_id * chunk + local_pos; the
   * element is rebuilt from its own sm byte and the stored exponent. */
  for (uint64_t k = 0; k < m->n_esc; ++k) {
    uint64_t cid = get_le32(payload + m->off_cid + 4 * k);
    uint64_t pos = get_le16(payload + m->off_lpos + 2 * k);
    uint64_t idx = cid * SZO_CHUNK + pos;
    if (pos >= SZO_CHUNK || idx >= m->n) return SZO_ERR_META;
    out[idx] = merge(payload[m->off_sm + idx], payload[m->off_ev + k]);
  }
  return SZO_OK;
}

void szo_to_p1_nibble_order(uint8_t* payload, const szo_meta* m) {
  for (uint64_t j = 0; j < m->n_pairs; ++j) {
    uint8_t b = payload[m->off_pk + j];
    payload[m->off_pk + j] = (uint8_t)(((b & 0x0Fu) << 4) | ((b >> 4) & 0x0Fu));
  }
}
