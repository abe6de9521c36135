/*
 * SplitZip BF16 codec -- CPU ORACLE (test infrastructure only).
 *
 * This is the plain, single-threaded, obviously-correct restatement of the
 * SplitZip method that the CUDA library is checked against.  Only the test
 * suite, the smoke check and the benchmark's CPU-baseline leg may load it; the
 * product path never does.  It shares no code, header, table or constant with
 * the CUDA library under weight_compression_codec_gb300/csrc.
 *
 * Sources (the pages the method is taken from):
 *   [P1] "splitzip_codec.py" (diffusers-dynamic-offloader SplitZip adapter):
 *        module docstring (bit split, payload layout), calibrate_codebook,
 *        PayloadMeta, _align4, assemble_payload, encode_torch, decode_torch.
 *   [P2] "docs/developer/splitzip.md": "What it does" (chunk = 1024),
 *        "Invariants common to both routes" item 1 (frozen wire format, LE).
 *
 * Conventions fixed where the pages are silent or disagree:
 *   - element 2i sits in the LOW nibble of pk[i] and element 2i+1 in the high
 *     nibble ([P1] encode_torch puts 2i in the high nibble; this codec uses the
 *     low-nibble order; szo_to_p1_nibble_order converts between the two);
 *   - an escaped element is stored in pk as code 0 ([P1] encode_torch masks
 *     the escape mark 16 with 0xF) and escapes are listed in ascending global
 *     index ([P1] encode_torch uses nonzero());
 *   - Top-16 ties are broken by ascending exponent value ([P1] leaves the
 *     order of an unstable descending argsort open);
 *   - n == 0 is accepted: coverage 1.0, no codes, empty payload.
 *
 * Parity status: every function here is pinned by tests/test_oracle_pins.py
 * (hand-worked golden payloads, all 65,536 bit patterns, library routines,
 * brute force and invariants) and tests/test_oracle_mutants.py.
 */
#ifndef SZ_ORACLE_H
#define SZ_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SZO_CHUNK 1024u   /* [P1] encode_torch chunk_size default; [P2] "chunk=1024" */
#define SZO_ESCAPE 16u    /* [P1] enc_lut_marked: value -> code or 16 (escape) */

typedef struct szo_codebook {
  uint8_t enc_lut[256];   /* exponent byte -> code 0..15, or 16 = escape  */
  uint8_t dec_lut[16];    /* code -> exponent byte; unused codes hold 0   */
  uint32_t n_top;         /* min(16, number of distinct exponents)        */
  uint64_t top_count;     /* elements whose exponent is one of the top    */
  double coverage;        /* top_count / n  (1.0 when n == 0)             */
} szo_codebook;

typedef struct szo_meta {
  uint64_t n, n_pairs, n_esc, comp_bytes;
  uint64_t off_pk, off_sm, off_cid, off_lpos, off_ev;
  uint32_t chunk_size;
  double coverage;
} szo_meta;

/* Status codes of the oracle. */
#define SZO_OK 0
#define SZO_ERR_CAPACITY 1
#define SZO_ERR_META 2

/* [P1] calibrate_codebook, first half: count every exponent byte
 * (x >> 7) & 0xFF of the n BF16 bit patterns. */
void szo_histogram(const uint16_t* x, uint64_t n, uint64_t hist[256]);

/* [P1] calibrate_codebook, second half: rank exponent values by count
 * (descending, ties by ascending value), keep the first min(16, distinct),
 * fill enc_lut / dec_lut and compute coverage = sum(top counts) / n. */
void szo_select(const uint64_t hist[256], uint64_t n, szo_codebook* cb);

/* szo_histogram followed by szo_select. */
void szo_calibrate(const uint16_t* x, uint64_t n, szo_codebook* cb);

/* [P1] PayloadMeta / assemble_payload: the section offsets and total size of
 * a payload of n elements with n_esc escapes.  coverage is copied in. */
void szo_layout(uint64_t n, uint64_t n_esc, double coverage, szo_meta* meta);

/* Number of elements whose exponent the codebook does not cover. */
uint64_t szo_count_escapes(const uint16_t* x, uint64_t n, const szo_codebook* cb);

/* [P1] encode_torch + assemble_payload: writes the whole payload (pads 0)
 * into out[0 .. meta->comp_bytes).  Returns SZO_ERR_CAPACITY (and writes
 * nothing) when capacity < comp_bytes. */
int szo_encode(const uint16_t* x, uint64_t n, const szo_codebook* cb,
               uint8_t* out, uint64_t capacity, szo_meta* meta);

/* [P1] decode_torch: dense reconstruction from (pk, sm, dec_lut), then every
 * escape in listed order overwrites its element with the stored exponent.
 * Returns SZO_ERR_META if the meta is inconsistent with its own n and n_esc
 * or an escape points outside [0, n). */
int szo_decode(const uint8_t* payload, const szo_meta* meta,
               const uint8_t dec_lut[16], uint16_t* out);

/* Rewrites the pk section of a payload in place so that element 2i moves to
 * the high nibble (the nibble order of [P1] encode_torch / decode_torch).
 * Applying it twice restores the input. */
void szo_to_p1_nibble_order(uint8_t* payload, const szo_meta* meta);

#ifdef __cplusplus
}
#endif
#endif
