/*
 * CPU oracle for the paged MLA KV-cache gather.
 *
 * TEST INFRASTRUCTURE ONLY. Only the tests, the smoke check and the
 * benchmark's CPU-baseline leg may load this file's library. The product path
 * (the CUDA library and its binding) never calls it and shares no code with it.
 *
 * What it computes follows "MLA cache gather scheduled per logical page"
 * (prhub.com.cn, vllm PR #51739), section "关键源码片段", the test
 * test_cp_gather_cache_mla_large_uneven_sequences: the expected output is the
 * concatenation over requests r of cache[block_table[r, p / B], p % B] for the
 * source positions p in [start_r, start_r + len_r). This file writes that
 * definition out as a per-request, per-token, per-element loop with 64-bit
 * integer arithmetic and nothing else: no pages, no tasks, no blocking.
 *
 * Output placement follows the page's mapper (same section, the
 * map_gather_page_task listing): request r owns output rows starting at
 * min(cu[r], T), its length is max(min(cu[r+1], T) - min(cu[r], T), 0), and
 * its source starts at seq_starts[r] (0 when seq_starts is absent).
 *
 * Readings where the page is silent:
 *  - The page's clamp decides each request's rows: a decrease of cu_seq_lens
 *    gives the request there no rows, and the other requests are copied as
 *    usual. What the page leaves open is a request with rows whose first row
 *    lies below an earlier boundary of cu_seq_lens (below cu[j] for some
 *    j < r, or below row 0): its rows would overlap rows written before, in
 *    an order the page does not fix, or run out of order. Such a request is
 *    skipped (bit 8); every other request is still copied.
 *  - A request with len > 0 and a negative start writes nothing (bit 4).
 *  - A token whose logical block is >= block_table_stride (bit 1) or whose
 *    physical block id is outside [0, num_blocks) (bit 2) is skipped; its
 *    output row is left untouched. The review section ("评论区精华") of the
 *    page reports exactly these two missing guards.
 *  - FP8 is OCP E4M3 ("fn": bias 7, no infinities, S.1111.111 is NaN).
 *    Dequant is one fp32 multiply by a per-tensor scale, then a single
 *    round-to-nearest-even into the destination type.
 *
 * Conversions are written from the format definitions (IEEE 754 binary16 and
 * binary32, bfloat16 as the top half of binary32, OCP 8-bit floating point
 * E4M3), not from any library's implementation.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

/* dtype codes of the oracle's own interface (numerically equal to the public
 * header's codes, which is an interface agreement, not shared code) */
enum { O_BF16 = 0, O_FP16 = 1, O_FP32 = 2, O_E4M3 = 3, O_U8 = 4 };

/* flag bits reported for invalid data */
enum { O_BAD_LOGICAL = 1, O_BAD_PHYS = 2, O_BAD_START = 4, O_BAD_CU = 8, O_BAD_TOKEN = 32 };

static int elem_bytes(int dt) {
  switch (dt) {
    case O_BF16: return 2;
    case O_FP16: return 2;
    case O_FP32: return 4;
    case O_E4M3: return 1;
    case O_U8: return 1;
    default: return 0;
  }
}

/* OCP E4M3: value = (-1)^s * 2^(e-7) * (1 + m/8) for e in 1..15 (except
 * e=15, m=7, which is NaN), and (-1)^s * 2^-6 * (m/8) for e = 0. Both are exact
 * in binary32: (8 + m) * 2^(e-10) and m * 2^-9. */
float pmg_oracle_e4m3_to_f32(uint8_t x) {
  const int s = (x >> 7) & 1;
  const int e = (x >> 3) & 0xF;
  const int m = x & 0x7;
  float mag;
  if (e == 15 && m == 7) {
    mag = NAN;
  } else if (e == 0) {
    mag = ldexpf((float)m, -9);
  } else {
    mag = ldexpf((float)(8 + m), e - 10);
  }
  return s ? -mag : mag;
}

/* bfloat16 is the high 16 bits of binary32 (exact). */
float pmg_oracle_bf16_to_f32(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

/* IEEE binary16: bias 15, 10 fraction bits, subnormals m * 2^-24. */
float pmg_oracle_f16_to_f32(uint16_t h) {
  const int s = (h >> 15) & 1;
  const int e = (h >> 10) & 0x1F;
  const int m = h & 0x3FF;
  float mag;
  if (e == 31) {
    mag = (m == 0) ? INFINITY : NAN;
  } else if (e == 0) {
    mag = ldexpf((float)m, -24);
  } else {
    mag = ldexpf((float)(1024 + m), e - 25);
  }
  return s ? -mag : mag;
}

/* binary32 -> bfloat16, round to nearest, ties to even. Done on the bit
 * pattern: adding 0x7FFF plus the lowest kept bit and truncating is the usual
 * integer form of round-half-even for a 16-bit truncation. NaN stays NaN
 * (quiet bit set, sign kept). */
uint16_t pmg_oracle_f32_to_bf16(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7FFFFFFFu) > 0x7F800000u) return (uint16_t)((u >> 16) | 0x0040u);
  const uint32_t lsb = (u >> 16) & 1u;
  u += 0x7FFFu + lsb;
  return (uint16_t)(u >> 16);
}

/* binary32 -> binary16, round to nearest, ties to even, with gradual
 * underflow and overflow to infinity. The binary32 significand (with its
 * hidden bit) is shifted right by the number of bits binary16 cannot hold at
 * this exponent and rounded on the dropped bits. */
uint16_t pmg_oracle_f32_to_f16(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  const uint16_t sign = (uint16_t)((u >> 16) & 0x8000u);
  const uint32_t a = u & 0x7FFFFFFFu;
  if (a > 0x7F800000u) return (uint16_t)(sign | 0x7E00u); /* NaN */
  if (a == 0x7F800000u) return (uint16_t)(sign | 0x7C00u); /* infinity */
  if (a < 0x00800000u) return sign; /* |f| < 2^-126: far below half of 2^-24 */
  const int e = (int)(a >> 23) - 127;                  /* unbiased exponent */
  const uint32_t sig = (a & 0x007FFFFFu) | 0x00800000u; /* 24-bit significand */
  if (e > 15) return (uint16_t)(sign | 0x7C00u);       /* >= 2^16: overflow */
  /* binary16 keeps 11 significand bits for normals (e >= -14) and fewer for
   * subnormals, whose unit is 2^-24 */
  const int shift = (e >= -14) ? 13 : 13 + (-14 - e);
  if (shift > 24) return sign; /* below 2^-25: rounds to zero */
  uint32_t q = sig >> shift;
  const uint32_t rem = sig & ((1u << shift) - 1u);
  const uint32_t half = 1u << (shift - 1);
  if (rem > half || (rem == half && (q & 1u))) q += 1u;
  if (e >= -14) {
    /* q in [2^10, 2^11]; q == 2^11 carries into the exponent */
    const uint32_t bits = ((uint32_t)(e + 15) << 10) + (q - 0x400u);
    if (bits >= 0x7C00u) return (uint16_t)(sign | 0x7C00u);
    return (uint16_t)(sign | bits);
  }
  /* subnormal: q in [0, 2^10]; q == 2^10 is the smallest normal */
  return (uint16_t)(sign | q);
}

/* Which (src, dst) pairs the gather defines: the same dtype is a byte copy;
 * FP8 E4M3 dequantises (with the scale) to bf16, fp16 or fp32; bf16 and fp16
 * widen to fp32 (no scale). */
int pmg_oracle_pair_supported(int src_dt, int dst_dt) {
  if (elem_bytes(src_dt) == 0 || elem_bytes(dst_dt) == 0) return 0;
  if (src_dt == dst_dt) return 1;
  if (src_dt == O_E4M3 && (dst_dt == O_BF16 || dst_dt == O_FP16 || dst_dt == O_FP32)) return 1;
  if ((src_dt == O_BF16 || src_dt == O_FP16) && dst_dt == O_FP32) return 1;
  return 0;
}

static void convert_one(const uint8_t* s, uint8_t* d, int src_dt, int dst_dt, float scale) {
  if (src_dt == dst_dt) {
    memcpy(d, s, (size_t)elem_bytes(src_dt));
    return;
  }
  float v;
  if (src_dt == O_E4M3) {
    v = pmg_oracle_e4m3_to_f32(s[0]) * scale; /* one binary32 multiply */
  } else if (src_dt == O_BF16) {
    uint16_t h;
    memcpy(&h, s, 2);
    v = pmg_oracle_bf16_to_f32(h);
  } else { /* O_FP16 */
    uint16_t h;
    memcpy(&h, s, 2);
    v = pmg_oracle_f16_to_f32(h);
  }
  if (dst_dt == O_FP32) {
    memcpy(d, &v, 4);
  } else if (dst_dt == O_BF16) {
    const uint16_t h = pmg_oracle_f32_to_bf16(v);
    memcpy(d, &h, 2);
  } else { /* O_FP16 */
    const uint16_t h = pmg_oracle_f32_to_f16(v);
    memcpy(d, &h, 2);
  }
}

/*
 * The gather. Strides are in elements of the array they index. Every pointer
 * is host memory. Returns the OR of the flag bits above (0 when every token
 * was copied), or -1 for a call the oracle does not define (unsupported dtype
 * pair, non-positive block or entry size, negative counts).
 */
int pmg_oracle_gather(const uint8_t* cache, int64_t cache_block_stride, int64_t cache_token_stride,
                      int64_t num_blocks, const int32_t* block_table, int64_t block_table_stride,
                      const int32_t* cu_seq_lens, const int32_t* seq_starts, int32_t num_reqs,
                      int64_t total_tokens, int32_t block_size, int32_t entry_size, int src_dtype,
                      int dst_dtype, float scale, uint8_t* dst, int64_t dst_token_stride) {
  if (!pmg_oracle_pair_supported(src_dtype, dst_dtype)) return -1;
  if (num_reqs < 0 || total_tokens < 0 || block_size < 1 || entry_size < 1) return -1;
  const int64_t es = elem_bytes(src_dtype);
  const int64_t ed = elem_bytes(dst_dtype);
  const int64_t T = total_tokens;
  const int64_t B = block_size;
  int flag = 0;

  /* the highest of row 0 and the clamped boundaries cu[0..r-1] */
  int64_t floor_row = 0;
  for (int32_t r = 0; r < num_reqs; ++r) {
    const int64_t ob = cu_seq_lens[r] < T ? cu_seq_lens[r] : T;
    const int64_t oe = cu_seq_lens[r + 1] < T ? cu_seq_lens[r + 1] : T;
    const int64_t len = oe - ob > 0 ? oe - ob : 0;
    const int64_t start = seq_starts ? (int64_t)seq_starts[r] : 0;
    const int64_t below = floor_row;
    if (ob > floor_row) floor_row = ob;
    if (len > 0 && ob < below) {
      flag |= O_BAD_CU;
      continue;
    }
    if (len > 0 && start < 0) {
      flag |= O_BAD_START;
      continue;
    }
    for (int64_t i = 0; i < len; ++i) {
      const int64_t p = start + i;
      const int64_t logical = p / B;
      const int64_t slot = p % B;
      if (logical >= block_table_stride) {
        flag |= O_BAD_LOGICAL;
        continue;
      }
      const int64_t phys = block_table[(int64_t)r * block_table_stride + logical];
      if (phys < 0 || phys >= num_blocks) {
        flag |= O_BAD_PHYS;
        continue;
      }
      const uint8_t* src = cache + (phys * cache_block_stride + slot * cache_token_stride) * es;
      uint8_t* d = dst + (ob + i) * dst_token_stride * ed;
      for (int64_t e = 0; e < entry_size; ++e) convert_one(src + e * es, d + e * ed, src_dtype, dst_dtype, scale);
    }
  }
  return flag;
}

/*
 * The per-token indexed gather of "indexer kernels take shape arguments at run
 * time" (prhub.com.cn, vllm PR #56153), section "关键源码片段", the kernel
 * _cp_gather_indexer_quant_cache_kernel: output token t
 * belongs to request b = token_to_seq[t]; its context position is t minus the
 * request's first output row cu_seq_lens[b]; the block table row b maps that
 * position's logical block to a physical block. Every index is bounds-checked
 * before use, the way that kernel masks its loads. A token whose request id is
 * outside [0, num_reqs), or that lies outside its request's rows
 * [cu[b], cu[b+1]), is skipped (bit 32); an out-of-row logical block (bit 1)
 * or physical id (bit 2) skips the token too. Skipped output rows are left
 * untouched. Returns the flag bits, or -1 outside the defined domain.
 */
int pmg_oracle_gather_tokens(const uint8_t* cache, int64_t cache_block_stride, int64_t cache_token_stride,
                             int64_t num_blocks, const int32_t* block_table, int64_t block_table_stride,
                             const int32_t* token_to_seq, const int32_t* cu_seq_lens, int32_t num_reqs,
                             int64_t num_tokens, int32_t block_size, int32_t entry_size, int src_dtype, int dst_dtype,
                             float scale, uint8_t* dst, int64_t dst_token_stride) {
  if (!pmg_oracle_pair_supported(src_dtype, dst_dtype)) return -1;
  if (num_reqs < 0 || num_tokens < 0 || block_size < 1 || entry_size < 1) return -1;
  const int64_t es = elem_bytes(src_dtype);
  const int64_t ed = elem_bytes(dst_dtype);
  int flag = 0;
  for (int64_t t = 0; t < num_tokens; ++t) {
    const int64_t b = token_to_seq[t];
    if (b < 0 || b >= num_reqs) {
      flag |= O_BAD_TOKEN;
      continue;
    }
    const int64_t first_row = cu_seq_lens[b];
    const int64_t end_row = cu_seq_lens[b + 1];
    if (t < first_row || t >= end_row) {
      flag |= O_BAD_TOKEN;
      continue;
    }
    const int64_t pos = t - first_row;
    const int64_t lblock = pos / block_size;
    const int64_t off = pos - lblock * block_size;
    if (lblock >= block_table_stride) {
      flag |= O_BAD_LOGICAL;
      continue;
    }
    const int64_t pb = block_table[b * block_table_stride + lblock];
    if (pb < 0 || pb >= num_blocks) {
      flag |= O_BAD_PHYS;
      continue;
    }
    const uint8_t* src = cache + (pb * cache_block_stride + off * cache_token_stride) * es;
    uint8_t* row = dst + t * dst_token_stride * ed;
    for (int64_t e = 0; e < entry_size; ++e) convert_one(src + e * es, row + e * ed, src_dtype, dst_dtype, scale);
  }
  return flag;
}
