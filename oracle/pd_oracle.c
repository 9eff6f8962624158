/*
 * pd_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, fp64 CPU statement of paged decode attention. Only the test
 * suite, the smoke check and the CPU-baseline leg of the benchmark may load
 * this file's library. The CUDA library shares no code, header or constant
 * with it, and neither one includes or calls the other.
 *
 * What it follows (opengfx1030/vllm-rdna pull request #33, "Paged split-K
 * decode", sections "Purpose" and "Test Result"):
 *   - the per-head decode computes, for each query token and head, a softmax
 *     over scale * q . k of the keys the token may see, weighted over V; the
 *     pull request checks its kernel schedule against a "one-shot fp64
 *     reference" -- pdo_decode_paged below is that one-shot definition;
 *   - the same section models the schedule as online softmax over tiles plus a
 *     split-K combine -- pdo_decode_paged_split below takes those steps, and
 *     pdo_combine is the combine on its own;
 *   - the "Test Plan" section names the behaviours: paged writer layout, empty
 *     rows give zeros, a caller-chosen scale, a sliding window, multi-token
 *     (speculative verify) queries with causal masking, and split decode.
 *
 * Readings where the page is silent (each one is listed with the others in
 * the design notes):
 *   - seq_lens[b] counts every cached key of sequence b, including the qlen
 *     query tokens themselves; query i sits at position p = L - qlen + i;
 *   - a window W > 0 keeps keys j with p - W + 1 <= j <= p; W <= 0 keeps all
 *     keys j <= p;
 *   - query head h reads KV head h / (Hq / Hkv);
 *   - Q and out are [B*qlen, Hq, D] with row b*qlen + i; the caches are
 *     [num_blocks, block_size, Hkv, D]; block_table is [B, max_blocks_per_seq];
 *   - fp8 KV holds OCP e4m3fn codes with one fp32 scale per cache: the value of
 *     a code c is decode(c) * k_scale (or v_scale); int8 KV holds signed
 *     two's-complement codes with the same per-cache scales ("Purpose": the
 *     fp8 and int8 decode wrappers share the body);
 *   - a row with no visible key is all zeros;
 *   - bfloat16 (not on the pages): a bfloat16 model keeps q and both caches
 *     in bfloat16 (kv_kind 3), or q in bfloat16 over e4m3fn or int8 caches
 *     (kv_kind 4 and 5); every value is still converted to fp64 exactly and
 *     the arithmetic is the same.
 *
 * Every value is converted to fp64 exactly and all arithmetic is fp64, in
 * key order, with no blocking beyond what each function states.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define PDO_OK 0
#define PDO_ERR_ARGS (-1)
#define PDO_ERR_BLOCK_ID (-2)
#define PDO_ERR_SEQ_LEN (-3)
#define PDO_ERR_NOMEM (-4)

typedef struct {
  int B, qlen, Hq, Hkv, D;
  int block_size, num_blocks, max_blocks_per_seq;
  int kv_kind;      /* 0: IEEE binary16 bit patterns; 1: e4m3fn bytes; 2: int8 codes;
                       3: bfloat16 bit patterns (q is then bfloat16 as well);
                       4, 5: e4m3fn bytes, int8 codes with bfloat16 q */
  double k_scale;   /* fp8 / int8: value = decode(code) * k_scale */
  double v_scale;
} pdo_dims;

/* IEEE 754 binary16: 1 sign, 5 exponent (bias 15), 10 fraction bits. */
double pdo_f16_to_f64(uint16_t h) {
  int sign = (h >> 15) & 1;
  int e = (h >> 10) & 0x1f;
  int f = h & 0x3ff;
  double v;
  if (e == 0)
    v = ldexp((double)f, -24); /* subnormal: f * 2^-10 * 2^-14 */
  else if (e == 31)
    v = f ? NAN : INFINITY;
  else
    v = ldexp((double)(1024 + f), e - 25); /* (1 + f/1024) * 2^(e-15) */
  return sign ? -v : v;
}

/* OCP 8-bit floating point, E4M3 "fn" variant: 1 sign, 4 exponent (bias 7),
 * 3 mantissa bits, no infinities, S.1111.111 is NaN, max normal 448. */
double pdo_e4m3fn_to_f64(uint8_t c) {
  int sign = (c >> 7) & 1;
  int e = (c >> 3) & 0xf;
  int m = c & 7;
  double v;
  if (e == 15 && m == 7)
    v = NAN;
  else if (e == 0)
    v = ldexp((double)m, -9); /* subnormal: m/8 * 2^-6 */
  else
    v = ldexp((double)(8 + m), e - 10); /* (1 + m/8) * 2^(e-7) */
  return sign ? -v : v;
}

/* bfloat16: 1 sign, 8 exponent (bias 127), 7 fraction bits -- the upper half
 * of an IEEE binary32. */
double pdo_bf16_to_f64(uint16_t h) {
  int sign = (h >> 15) & 1;
  int e = (h >> 7) & 0xff;
  int f = h & 0x7f;
  double v;
  if (e == 0)
    v = ldexp((double)f, -133); /* subnormal: f/128 * 2^-126 */
  else if (e == 255)
    v = f ? NAN : INFINITY;
  else
    v = ldexp((double)(128 + f), e - 134); /* (1 + f/128) * 2^(e-127) */
  return sign ? -v : v;
}

/* Signed 8-bit two's-complement code. */
double pdo_i8_to_f64(uint8_t c) { return (double)(int8_t)c; }

/* Value of element x of (block, slot, kv head) in a K or V cache. */
static double cache_at(const pdo_dims* d, const void* cache, double fp8_scale, long blk,
                       int slot, int kh, int x) {
  long idx = ((blk * d->block_size + slot) * (long)d->Hkv + kh) * d->D + x;
  if (d->kv_kind == 1 || d->kv_kind == 4)
    return pdo_e4m3fn_to_f64(((const uint8_t*)cache)[idx]) * fp8_scale;
  if (d->kv_kind == 2 || d->kv_kind == 5) return pdo_i8_to_f64(((const uint8_t*)cache)[idx]) * fp8_scale;
  if (d->kv_kind == 3) return pdo_bf16_to_f64(((const uint16_t*)cache)[idx]);
  return pdo_f16_to_f64(((const uint16_t*)cache)[idx]);
}

/* Element x of a query row (fp16, or bfloat16 for kv_kind 3, 4 and 5). */
static double q_at(const pdo_dims* d, const uint16_t* q, long rho, int x) {
  uint16_t bits = q[rho * d->D + x];
  return d->kv_kind >= 3 ? pdo_bf16_to_f64(bits) : pdo_f16_to_f64(bits);
}

/* Visible key range [*lo, *hi] of query token i of a sequence of length L.
 * Returns 0 when the token sees no key. */
static int visible_range(int L, int qlen, int i, int window, long* lo, long* hi) {
  long p = (long)L - qlen + i;
  if (L <= 0 || p < 0) return 0;
  long first = 0;
  if (window > 0 && p - window + 1 > 0) first = p - window + 1;
  *lo = first;
  *hi = p;
  return 1;
}

static int check_args(const pdo_dims* d) {
  if (!d || d->B < 0 || d->qlen < 1 || d->Hq < 1 || d->Hkv < 1 || d->D < 1 ||
      d->Hq % d->Hkv != 0 || d->block_size < 1 || d->num_blocks < 0 || d->max_blocks_per_seq < 0)
    return PDO_ERR_ARGS;
  return PDO_OK;
}

/* Physical block of logical key j of sequence b, or -1 when the table entry
 * is out of range. */
static long phys_block(const pdo_dims* d, const int32_t* block_table, int b, long j) {
  long lb = j / d->block_size;
  int32_t blk = block_table[(long)b * d->max_blocks_per_seq + lb];
  if (blk < 0 || blk >= d->num_blocks) return -1;
  return blk;
}

/*
 * One-shot definition. For every output row rho in [row_begin, row_end),
 * rho = (b*qlen + i)*Hq + h:
 *     s_j   = scale * sum_x q[x] * K_j[x]            for visible keys j
 *     out   = sum_j exp(s_j - M) V_j / sum_j exp(s_j - M),  M = max_j s_j
 * and out = 0 when no key is visible. q is fp16 bit patterns.
 */
int pdo_decode_paged(const pdo_dims* d, const uint16_t* q, const void* k_cache,
                     const void* v_cache, const int32_t* block_table, const int32_t* seq_lens,
                     double scale, int window, long row_begin, long row_end, double* out) {
  if (check_args(d)) return PDO_ERR_ARGS;
  const int D = d->D, G = d->Hq / d->Hkv;
  long cap = (long)d->max_blocks_per_seq * d->block_size;
  double* s = NULL;
  double* qv = (double*)malloc(sizeof(double) * D);
  if (!qv) return PDO_ERR_NOMEM;
  int rc = PDO_OK;
  for (long rho = row_begin; rho < row_end && rc == PDO_OK; ++rho) {
    int h = (int)(rho % d->Hq);
    long tok = rho / d->Hq;
    int b = (int)(tok / d->qlen), i = (int)(tok % d->qlen);
    int kh = h / G;
    double* o = out + rho * D;
    for (int x = 0; x < D; ++x) o[x] = 0.0;
    int L = seq_lens[b];
    if (L < 0 || L > cap) { rc = PDO_ERR_SEQ_LEN; break; }
    long lo, hi;
    if (!visible_range(L, d->qlen, i, window, &lo, &hi)) continue;
    long n = hi - lo + 1;
    s = (double*)realloc(s, sizeof(double) * n);
    if (!s) { rc = PDO_ERR_NOMEM; break; }
    for (int x = 0; x < D; ++x) qv[x] = q_at(d, q, rho, x);
    double M = -INFINITY;
    for (long j = lo; j <= hi; ++j) {
      long blk = phys_block(d, block_table, b, j);
      if (blk < 0) { rc = PDO_ERR_BLOCK_ID; break; }
      int slot = (int)(j % d->block_size);
      double dot = 0.0;
      for (int x = 0; x < D; ++x) dot += qv[x] * cache_at(d, k_cache, d->k_scale, blk, slot, kh, x);
      s[j - lo] = scale * dot;
      if (s[j - lo] > M) M = s[j - lo];
    }
    if (rc != PDO_OK) break;
    double l = 0.0;
    for (long j = lo; j <= hi; ++j) {
      long blk = phys_block(d, block_table, b, j);
      int slot = (int)(j % d->block_size);
      double w = exp(s[j - lo] - M);
      l += w;
      for (int x = 0; x < D; ++x) o[x] += w * cache_at(d, v_cache, d->v_scale, blk, slot, kh, x);
    }
    for (int x = 0; x < D; ++x) o[x] /= l;
  }
  free(s);
  free(qv);
  return rc;
}

/*
 * Split-K combine of S partials for each of `rows` rows. Partial s of row r is
 * (m[r*S+s], l[r*S+s], O[(r*S+s)*D : +D]) with m the largest score of the
 * chunk (natural-log units), l = sum exp(s_j - m) and O = sum exp(s_j - m) V_j
 * over the chunk; an empty chunk has m = -inf, l = 0, O = 0.
 *     M = max_s m_s,  w_s = exp(m_s - M) (0 for an empty chunk),
 *     out = sum_s w_s O_s / sum_s w_s l_s,   out = 0 when every chunk is empty.
 */
int pdo_combine(long rows, int S, int D, const double* m, const double* l, const double* O,
                double* out) {
  if (rows < 0 || S < 1 || D < 1) return PDO_ERR_ARGS;
  for (long r = 0; r < rows; ++r) {
    double* o = out + r * D;
    for (int x = 0; x < D; ++x) o[x] = 0.0;
    double M = -INFINITY;
    for (int s = 0; s < S; ++s)
      if (m[r * S + s] > M) M = m[r * S + s];
    if (M == -INFINITY) continue;
    double L = 0.0;
    for (int s = 0; s < S; ++s) {
      double ms = m[r * S + s];
      double w = (ms == -INFINITY) ? 0.0 : exp(ms - M);
      L += w * l[r * S + s];
      for (int x = 0; x < D; ++x) o[x] += w * O[(r * S + s) * (long)D + x];
    }
    if (L > 0.0)
      for (int x = 0; x < D; ++x) o[x] /= L;
    else
      for (int x = 0; x < D; ++x) o[x] = 0.0;
  }
  return PDO_OK;
}

/*
 * Split mode: the same result reached the way the pull request's numeric model
 * reaches it. For each sequence, the blocks that hold visible keys of any of
 * its query tokens, from the block of the first visible key of token 0 to the
 * block of key L-1, are cut into S contiguous chunks of ceil(n/S) blocks (the
 * last chunks may be empty). Each chunk is walked block by block with online
 * softmax -- running max m, running sum l, running O rescaled by exp(m_old -
 * m_new) whenever the max grows -- then the S chunk partials are merged by
 * pdo_combine. Keys outside a token's visible range are skipped.
 * If m_out/l_out/O_out are non-NULL the per-chunk partials are stored there
 * ([rows][S], [rows][S], [rows][S][D], rows indexed as in pdo_decode_paged).
 */
int pdo_decode_paged_split(const pdo_dims* d, const uint16_t* q, const void* k_cache,
                           const void* v_cache, const int32_t* block_table,
                           const int32_t* seq_lens, double scale, int window, int S,
                           long row_begin, long row_end, double* out, double* m_out,
                           double* l_out, double* O_out) {
  if (check_args(d) || S < 1) return PDO_ERR_ARGS;
  const int D = d->D, G = d->Hq / d->Hkv, bs = d->block_size;
  long cap = (long)d->max_blocks_per_seq * bs;
  double* qv = (double*)malloc(sizeof(double) * D);
  double* pm = (double*)malloc(sizeof(double) * S);
  double* pl = (double*)malloc(sizeof(double) * S);
  double* pO = (double*)malloc(sizeof(double) * S * (long)D);
  if (!qv || !pm || !pl || !pO) { free(qv); free(pm); free(pl); free(pO); return PDO_ERR_NOMEM; }
  int rc = PDO_OK;
  for (long rho = row_begin; rho < row_end && rc == PDO_OK; ++rho) {
    int h = (int)(rho % d->Hq);
    long tok = rho / d->Hq;
    int b = (int)(tok / d->qlen), i = (int)(tok % d->qlen);
    int kh = h / G;
    int L = seq_lens[b];
    if (L < 0 || L > cap) { rc = PDO_ERR_SEQ_LEN; break; }
    for (int s = 0; s < S; ++s) {
      pm[s] = -INFINITY;
      pl[s] = 0.0;
      for (int x = 0; x < D; ++x) pO[(long)s * D + x] = 0.0;
    }
    long lo = 0, hi = -1;
    int any = visible_range(L, d->qlen, i, window, &lo, &hi);
    /* Block range of the sequence: token 0's first visible key to key L-1. */
    long lo0 = 0, hi0 = -1;
    long n_blocks = 0, first_block = 0;
    if (L > 0) {
      long p0 = (long)L - d->qlen;
      lo0 = (window > 0 && p0 - window + 1 > 0) ? p0 - window + 1 : 0;
      hi0 = L - 1;
      first_block = lo0 / bs;
      n_blocks = hi0 / bs - first_block + 1;
    }
    long chunk = (n_blocks + S - 1) / S;
    for (int x = 0; x < D; ++x) qv[x] = q_at(d, q, rho, x);
    for (int s = 0; s < S && any; ++s) {
      long cb0 = first_block + (long)s * chunk;
      long cb1 = cb0 + chunk;
      if (cb1 > first_block + n_blocks) cb1 = first_block + n_blocks;
      double m = -INFINITY, l = 0.0;
      double* O = pO + (long)s * D;
      for (long lb = cb0; lb < cb1 && rc == PDO_OK; ++lb) {
        /* one block of keys: [lb*bs, lb*bs + bs) */
        for (long j = lb * bs; j < (lb + 1) * bs; ++j) {
          if (j < lo || j > hi) continue;
          long blk = phys_block(d, block_table, b, j);
          if (blk < 0) { rc = PDO_ERR_BLOCK_ID; break; }
          int slot = (int)(j % bs);
          double dot = 0.0;
          for (int x = 0; x < D; ++x) dot += qv[x] * cache_at(d, k_cache, d->k_scale, blk, slot, kh, x);
          double sj = scale * dot;
          if (sj > m) {
            double a = (m == -INFINITY) ? 0.0 : exp(m - sj);
            l *= a;
            for (int x = 0; x < D; ++x) O[x] *= a;
            m = sj;
          }
          double w = exp(sj - m);
          l += w;
          for (int x = 0; x < D; ++x) O[x] += w * cache_at(d, v_cache, d->v_scale, blk, slot, kh, x);
        }
      }
      pm[s] = m;
      pl[s] = l;
    }
    if (rc != PDO_OK) break;
    if (m_out)
      for (int s = 0; s < S; ++s) m_out[rho * S + s] = pm[s];
    if (l_out)
      for (int s = 0; s < S; ++s) l_out[rho * S + s] = pl[s];
    if (O_out) memcpy(O_out + rho * S * (long)D, pO, sizeof(double) * S * (long)D);
    pdo_combine(1, S, D, pm, pl, pO, out + rho * D);
  }
  free(qv);
  free(pm);
  free(pl);
  free(pO);
  return rc;
}

/*
 * Quantisers of the paged KV-cache writer. The test plan of the pull request
 * ("Test Plan": the writer-layout cell) checks that the decode reads back what
 * the cache writer stored; the writer's arithmetic is not spelled out there,
 * so these follow the plain reading: a new value x (fp16) is divided by the
 * cache's scale in IEEE single precision, and the quotient t is stored as the
 * nearest code.
 */

/* e4m3fn code nearest to t, found by trying every finite code: ties go to the
 * even code, anything beyond 448 in magnitude (infinities included) saturates
 * to +-448, the sign of t (zero included) is kept, NaN gives 0x7F. */
uint8_t pdo_e4m3fn_encode(float t) {
  if (isnan(t)) return 0x7f;
  uint8_t sign = signbit(t) ? 0x80 : 0x00;
  double a = fabs((double)t);
  if (isinf(t)) return sign | 0x7e;
  int best = 0;
  double best_d = INFINITY;
  for (int c = 0; c <= 0x7e; ++c) {
    double d = fabs(pdo_e4m3fn_to_f64((uint8_t)c) - a);
    if (d < best_d || (d == best_d && (c & 1) == 0)) {
      best = c;
      best_d = d;
    }
  }
  return sign | (uint8_t)best;
}

/* Nearest integer to t, ties to even, clamped to [-127, 127]; NaN gives 0. */
int8_t pdo_i8_encode(float t) {
  if (isnan(t)) return 0;
  double v = (double)t;
  if (v >= 127.0) return 127;
  if (v <= -127.0) return -127;
  double f = floor(v);
  double frac = v - f;
  double r;
  if (frac > 0.5)
    r = f + 1.0;
  else if (frac < 0.5)
    r = f;
  else
    r = (fmod(f, 2.0) == 0.0) ? f : f + 1.0;
  return (int8_t)r;
}

/*
 * Paged KV-cache writer. New token t in [0, T) carries k_new[t] and v_new[t]
 * ([T, Hkv, D] fp16 bit patterns) and a slot slot_mapping[t] in the cache:
 * block slot / block_size, offset slot % block_size. A negative slot marks a
 * padding token and writes nothing. For every KV head h and dim x of a token:
 *   fp16 cache:  K[block][offset][h][x] = k_new[t][h][x]        (bit copy;
 *                likewise a bfloat16 cache from bfloat16 input)
 *   fp8 cache:   pdo_e4m3fn_encode(fp32(k_new) / fp32(k_scale))
 *   int8 cache:  pdo_i8_encode(fp32(k_new) / fp32(k_scale))
 * and likewise V with v_scale. A slot at or beyond num_blocks * block_size
 * writes nothing and makes the call return PDO_ERR_BLOCK_ID once every other
 * token has been written.
 */
int pdo_write_kv_cache(const pdo_dims* d, const uint16_t* k_new, const uint16_t* v_new,
                       const int64_t* slot_mapping, long T, void* k_cache, void* v_cache) {
  if (!d || T < 0 || d->Hkv < 1 || d->D < 1 || d->block_size < 1 || d->num_blocks < 0 ||
      d->kv_kind < 0 || d->kv_kind > 5)
    return PDO_ERR_ARGS;
  const long row = (long)d->Hkv * d->D;
  const int64_t cap = (int64_t)d->num_blocks * d->block_size;
  const float ks = (float)d->k_scale, vs = (float)d->v_scale;
  int rc = PDO_OK;
  for (long t = 0; t < T; ++t) {
    int64_t slot = slot_mapping[t];
    if (slot < 0) continue;
    if (slot >= cap) { rc = PDO_ERR_BLOCK_ID; continue; }
    long blk = (long)(slot / d->block_size), off = (long)(slot % d->block_size);
    long dst = (blk * d->block_size + off) * row;
    for (long e = 0; e < row; ++e) {
      uint16_t kx = k_new[t * row + e], vx = v_new[t * row + e];
      if (d->kv_kind == 0 || d->kv_kind == 3) {  /* 16-bit caches: the input's bits */
        ((uint16_t*)k_cache)[dst + e] = kx;
        ((uint16_t*)v_cache)[dst + e] = vx;
      } else {
        /* new tokens in fp16, or bfloat16 for the bfloat16-q kinds 4 and 5 */
        const int b16 = d->kv_kind >= 4;
        float kq = (float)(b16 ? pdo_bf16_to_f64(kx) : pdo_f16_to_f64(kx)) / ks;
        float vq = (float)(b16 ? pdo_bf16_to_f64(vx) : pdo_f16_to_f64(vx)) / vs;
        if (d->kv_kind == 1 || d->kv_kind == 4) {
          ((uint8_t*)k_cache)[dst + e] = pdo_e4m3fn_encode(kq);
          ((uint8_t*)v_cache)[dst + e] = pdo_e4m3fn_encode(vq);
        } else {
          ((uint8_t*)k_cache)[dst + e] = (uint8_t)pdo_i8_encode(kq);
          ((uint8_t*)v_cache)[dst + e] = (uint8_t)pdo_i8_encode(vq);
        }
      }
    }
  }
  return rc;
}
