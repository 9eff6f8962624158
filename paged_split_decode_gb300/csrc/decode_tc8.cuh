// decode_tc8.cuh -- paged decode attention for e4m3 caches on the 5th-generation
// tensor cores (tcgen05, accumulators in tensor memory), for units with many
// query rows per KV head (G * qlen up to 32: speculative verify, wide GQA).
//
// Same method and work split as decode_kernel.cuh (the per-head paged decode
// of opengfx1030/vllm-rdna pull request #33, "Purpose"; split-K pieces merged
// by the split-combine kernel), different engine:
//  * A unit is (sequence, KV head); its visible 16-key tiles are cut into
//    pieces by the balanced split (work_next). Within a piece, 8 consecutive
//    tiles form a 128-key block. Two producer warps TMA-load the K and the V
//    rows of each block (128-byte swizzled, the layout the tensor cores read)
//    into rings of block stages, all boxes of a block at once.
//  * One thread issues tcgen05.mma kind::f8f6f4 on the e4m3 codes themselves:
//    S^T[128 keys x 96] = K Q^T into tensor memory, and later O^T[D x 96] +=
//    V^T P^T. The K and V codes are never widened.
//  * q (fp16) is scaled per row by a power of two and split exactly into three
//    e4m3 terms, q = t1 + t2 + t3 (see split3_e4m3); the terms are stacked on
//    the N side (3 x 32 rows) and their products summed when S^T is read. The
//    softmax weights are split the same way and stacked on N for P.V; the
//    three O^T accumulators are summed at the end of a piece.
//  * Softmax warps in NG groups of four (NG = the unit's 8-row tiles, 2 to
//    4): thread i of a group owns TMEM lane i (key i of a block), and group g
//    owns query rows 8 g .. 8 g + 7 (their maxima, sums and O^T columns), so
//    the groups never wait on each other and no group works on padding rows
//    beyond its tile. They read S^T, mask, take the per-row block maximum
//    (warp transpose-reduce and a shared exchange), form the weights against a
//    running maximum that is only raised when the block maximum exceeds it by
//    more than 2^4 (then the O^T accumulator is rescaled in tensor memory), and
//    write P^T: each key's thread stores its 8 row weights per term as one
//    8-byte piece of a 32-byte row of an MN-major operand (32-byte swizzle).
//    V^T is read by the product straight from the ring as an MN-major operand
//    (each 128-byte key row is 128 consecutive dims). Keys past the sequence
//    end or outside the piece get -inf scores and their V rows are zeroed in
//    the ring.
//  * K and V have rings of their own: a K stage is released when S^T is
//    computed, a V stage when the P.V product that reads it completes.
//  * At the end of a piece the warps read O^T (one output dim per thread) and
//    write fp16 rows (unit done in one piece) or the fp32 (m, l, O) partial.
//  * Every wait is bounded; after a timeout each role stops waiting and
//    issuing but keeps the softmax warps' named-barrier sequence, so the CTA
//    always reaches its exit, where the tensor memory is freed.
#pragma once
#include "launch.h"
#include "tc5.cuh"

namespace pd {

template <int D_, bool QB_ = false, int NG_ = 4>
struct Tc8 {
  static constexpr int D = D_;
  static constexpr bool QB = QB_;                   // q and out in bfloat16 (else fp16)
  static constexpr int NG = NG_;                    // softmax groups = 8-row tiles of a unit (1 to 4)
  static constexpr int kSlabs = D / 128;            // 128-byte slabs of one e4m3 key row
  static constexpr int kBlkTiles = 8;               // 16-key tiles per 128-key block
  static constexpr int kSlabBlk = 128 * 128;        // one slab of a block: [128 keys][128 B]
  static constexpr int kKBlk = kSlabs * kSlabBlk;   // K (or V) of one block
  static constexpr int NBK = D == 256 ? 2 : 4;      // K ring stages
  static constexpr int NBV = D == 256 ? 3 : 5;      // V ring stages (held until P.V completes)
  static constexpr int kTileBox = 16 * 128;         // one TMA box: 16 keys x 128 bytes
  static constexpr int kN = 32;                     // query rows per unit on the N side
  static constexpr int kNT = 3 * kN;                // N of both products: three terms x 32 rows
  static constexpr int kQSlab = kNT * 128;          // q operand, one slab: [term][32 rows][128 B]
  static constexpr int kQBytes = kSlabs * kQSlab;
  static constexpr int kPtTerm = 128 * kN;          // one P^T term: [128 keys][32 rows], MN-major
  static constexpr int kGroupRows = 8;              // query rows per softmax group
  static constexpr int kSoftThreads = 128 * NG;     // softmax warps 0 .. 4 NG - 1
  static constexpr int kThreads = kSoftThreads + 96;  // then the K and V producers and the MMA warp
  static constexpr int kProducerWarp = 4 * NG, kMmaWarp = 4 * NG + 2;
  static constexpr int kBarAll = NG + 1;            // named barrier of every softmax thread (1..NG: groups)
  static constexpr int kTmemCols = 512;             // S^T x2 (2 x 96), O^T (kSlabs x 96)
  static constexpr int kColS = 0, kColO = 2 * kNT;
  static constexpr uint32_t kIdescS = idesc_e4m3(128, kNT);               // K-major A and B
  static constexpr uint32_t kIdescO = idesc_e4m3(128, kNT) | (3u << 15);  // A (V^T), B (P^T) MN-major
  static constexpr float kRaise = 4.f;              // running max raised past this gap (log2)
  // Balanced split: a piece's fixed cost (q set-up, pipeline refill, epilogue)
  // is charged as this many 16-key tiles to the start of every unit (measured
  // on the qlen=3 verify shape: 0 / 8 / 16 / 24 / 32 tiles -> 44.5 / 43.3 /
  // 41.7 / 40.2 / 40.2 us per step).
  static constexpr int kUnitCost = 24;
  static constexpr float kBias = 4.f;               // weights are 2^(x - m + kBias) <= 2^8

  static constexpr int kOffV = NBK * kKBlk;
  static constexpr int kOffQ = kOffV + NBV * kKBlk;
  static constexpr int kOffPt = kOffQ + kQBytes;
  static constexpr int kOffRed = kOffPt + 3 * kPtTerm;     // float [NG groups][4 warps][8 rows]
  static constexpr int kRowWords = 7 * 32;                 // row state: 7 arrays of 32 words
  static constexpr int kOffRow = kOffRed + NG * 4 * kGroupRows * 4;
  // Cluster merge (a fixed split whose pieces are the CTAs of one cluster):
  // each CTA stages its partial (m, l) here and its partial O rows [32][D]
  // fp32 at offset 0, over the K ring, which is idle once the piece is done.
  static constexpr int kOffStageMl = kOffRow + kRowWords * 4;  // float2 [32 rows]
  static constexpr int kOffBars = kOffStageMl + 32 * 8;
  static constexpr int kBars = 2 * NBK + 2 * NBV + 8;
  static constexpr int kOffTmem = kOffBars + kBars * 8;
  static constexpr int kOffPre = kOffTmem + 16;
  static constexpr int kSmemBytes = kOffPre + (kMaxAutoB + 1) * 4 + 1024;  // + alignment slack
  static_assert(D == 128 || D == 256, "head size 128 or 256");
  static_assert(NG >= 1 && NG <= 4, "one to four 8-row tiles per unit");
  static_assert(kGroupRows * NG <= kN, "rows of every group on the N side");
  static_assert(kOffV % 1024 == 0 && kOffQ % 1024 == 0 && kOffPt % 1024 == 0 && kQSlab % 1024 == 0 &&
                    kPtTerm % 1024 == 0,
                "tensor-core operands start on 1024-byte swizzle atoms");
  static_assert(kSmemBytes <= 227 * 1024, "one CTA per SM");
  static_assert(kN * D * 4 <= NBK * kKBlk, "the staged O rows fit over the K ring");
};

// A 16-bit pair (fp16, or bfloat16 with QB) as two floats, exactly.
template <bool QB>
__device__ __forceinline__ float2 pair_to_float2(uint32_t w) {
  if constexpr (QB) return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
  else return __half22float2(*reinterpret_cast<const __half2*>(&w));
}

// An fp16 pair to two e4m3fn codes (low half -> low byte), round to nearest
// even, saturating at +-448.
__device__ __forceinline__ uint32_t half2_to_e4m3x2(uint32_t h) {
  uint16_t d;
  asm("cvt.rn.satfinite.e4m3x2.f16x2 %0, %1;" : "=h"(d) : "r"(h));
  return d;
}
// An fp16 pair x as three e4m3 code pairs whose values add up to x: t1 =
// e4m3(x), t2 = e4m3(x - t1), t3 = e4m3(x - t1 - t2) (codes in the low 16
// bits). Each difference is exact in fp16 (a multiple of x's last place, at
// most half of t1's step), and three 4-bit significands cover fp16's 11 bits,
// so the sum is x exactly unless a remainder falls below e4m3's subnormal
// step 2^-9 (then the error is at most 2^-10). |x| <= 448.
__device__ __forceinline__ void split3_e4m3(uint32_t x, uint32_t& t1, uint32_t& t2, uint32_t& t3) {
  t1 = half2_to_e4m3x2(x);
  const uint32_t f1 = e4m3x2_to_half2(static_cast<uint16_t>(t1));
  const __half2 r1 = __hsub2(*reinterpret_cast<const __half2*>(&x), *reinterpret_cast<const __half2*>(&f1));
  const uint32_t r1u = *reinterpret_cast<const uint32_t*>(&r1);
  t2 = half2_to_e4m3x2(r1u);
  const uint32_t f2 = e4m3x2_to_half2(static_cast<uint16_t>(t2));
  const __half2 r2 = __hsub2(r1, *reinterpret_cast<const __half2*>(&f2));
  t3 = half2_to_e4m3x2(*reinterpret_cast<const uint32_t*>(&r2));
}

// Row state arrays in shared memory (32 entries each).
// kRowCf (a per-row score offset) is used by the int8 kernel only.
enum { kRowFsl = 0, kRowMu = 1, kRowAl = 2, kRowLo = 3, kRowHi = 4, kRowL = 5, kRowFlag = 6, kRowCf = 7 };
// Barriers: fullK[NBK], emptyK[NBK], fullV[NBV], emptyV[NBV], then these.
enum { kBarSFull = 0, kBarSEmpty = 2, kBarPFull = 4, kBarPvDone = 5, kBarQFull = 6, kBarFinal = 7 };

// N values (8, 16 or 32), one per row, held by every lane of a warp -> lane
// l holds the reduction of row l % N over the 32 lanes (log2 N butterfly
// rounds exchanging half of the remaining values, then the lane groups).
template <bool MAX, int N>
__device__ __forceinline__ float warp_transpose_reduce(float (&v)[N], int lane) {
  static_assert(N == 8 || N == 16 || N == 32, "8, 16 or 32 rows");
#pragma unroll
  for (int w = N / 2; w >= 1; w >>= 1) {
    const bool up = (lane & w) != 0;
#pragma unroll
    for (int k = 0; k < w; ++k) {
      const float send = up ? v[k] : v[k + w];
      const float keep = up ? v[k + w] : v[k];
      const float recv = __shfl_xor_sync(0xffffffffu, send, w);
      v[k] = MAX ? fmaxf(keep, recv) : keep + recv;
    }
  }
  float r = v[0];
#pragma unroll
  for (int o = N; o < 32; o <<= 1) {
    const float other = __shfl_xor_sync(0xffffffffu, r, o);
    r = MAX ? fmaxf(r, other) : r + other;
  }
  return r;
}

// The next piece with visible tiles for the softmax warps (thread index < NST);
// pieces with nothing visible are finished on the spot: their rows are written
// as zeros (such a unit is never split).
template <class T>
__device__ __forceinline__ bool tc_next_piece(const DecodeParams& p, const int* s_pre, WorkIter& it, Piece& out) {
  constexpr int D = T::D;
  while (work_next(p, s_pre, it, out)) {
    if (out.ntiles > 0) return true;
    for (int item = threadIdx.x; item < out.R * (D / 8); item += T::kSoftThreads) {
      const int r = item / (D / 8), dc = item % (D / 8);
      const int i = r / p.G, hl = r % p.G;
      *reinterpret_cast<uint4*>(p.out + (static_cast<long long>(out.q0 + i) * p.Hq + out.kh * p.G + hl) * D +
                                dc * 8) = make_uint4(0u, 0u, 0u, 0u);
    }
  }
  return false;
}

// Scores of key key0 + key for the rows rb .. rb + 7 in the log2 domain: the
// products times the row factors fs (plus the row offsets cf with OFF); -inf
// for keys not loaded (key >= nvalid) or outside a row's visible range [lo, hi]
// (causal end and window). A block whose keys all lie inside every row's range
// skips the per-row test.
template <class T, bool OFF = false>
__device__ __forceinline__ void tc_scale_mask(float (&x)[8], const float (&fs)[8], const float (&cf)[8], int key0,
                                              int nvalid, const Piece& pc, const int* ri, int rb, int key) {
  constexpr int NR = T::kGroupRows;
  auto scaled = [&](int r) { return OFF ? fmaf(x[r], fs[r], cf[r]) : x[r] * fs[r]; };
  const bool interior = nvalid == 128 && key0 >= pc.tile_lo_all && key0 + 127 <= pc.tile_hi_all;
  if (interior) {
#pragma unroll
    for (int r = 0; r < NR; ++r) x[r] = scaled(r);
  } else {
    const int j = key0 + key;
    const bool loaded = key < nvalid;
#pragma unroll
    for (int r = 0; r < NR; ++r)
      x[r] = (loaded && j >= ri[kRowLo * 32 + rb + r] && j <= ri[kRowHi * 32 + rb + r]) ? scaled(r) : -INFINITY;
  }
}

// Running maximum of a softmax group's 8 rows (rows 8 g .. 8 g + 7, the
// group's named barrier 1 + g), raised to the block maximum only where that
// exceeds it by more than 2^kRaise. Most blocks raise nothing: one OR-barrier
// tells, and only then are the block maxima reduced (warp transpose-reduce and
// a shared exchange). On return mu holds the rows' maxima; the result says
// whether any row was raised, its factor 2^(old - new) then in kRowAl.
template <class T>
__device__ __forceinline__ bool tc_raise_max(const float (&x)[8], float (&mu)[8], float* rf, int* ri, float* red,
                                             int g, int warp, int lane) {
  constexpr int NR = T::kGroupRows;
  const int rb = NR * g, bid = 1 + g;
  auto load8 = [&](const float* src) {
#pragma unroll
    for (int k = 0; k < NR / 4; ++k) {
      const float4 f = reinterpret_cast<const float4*>(src)[k];
      mu[4 * k] = f.x; mu[4 * k + 1] = f.y; mu[4 * k + 2] = f.z; mu[4 * k + 3] = f.w;
    }
  };
  load8(rf + kRowMu * 32 + rb);
  bool upd = false;
#pragma unroll
  for (int r = 0; r < NR; ++r) upd |= x[r] > mu[r] + T::kRaise;
  if (!bar_red_or(bid, 128, upd)) return false;
  {
    float v[NR];
#pragma unroll
    for (int r = 0; r < NR; ++r) v[r] = x[r];
    const float m = warp_transpose_reduce<true, NR>(v, lane);
    if (lane < NR) red[(warp & 3) * NR + lane] = m;
  }
  named_bar_sync(bid, 128);
  if ((warp & 3) == 0 && lane < NR) {
    const float mx = fmaxf(fmaxf(red[lane], red[NR + lane]), fmaxf(red[2 * NR + lane], red[3 * NR + lane]));
    const float m0 = rf[kRowMu * 32 + rb + lane];
    float nmu = m0, al = 1.f;
    if (mx > m0 + T::kRaise) {
      nmu = mx;
      al = (m0 == -INFINITY) ? 0.f : ex2(m0 - mx);
    }
    rf[kRowMu * 32 + rb + lane] = nmu;
    rf[kRowAl * 32 + rb + lane] = al;
    const bool any = __any_sync((1u << NR) - 1u, al != 1.f);
    if (lane == 0) ri[kRowFlag * 32 + g] = any ? 1 : 0;
  }
  named_bar_sync(bid, 128);
  load8(rf + kRowMu * 32 + rb);
  return ri[kRowFlag * 32 + g] != 0;
}

// End of a piece for softmax group g: the rows' weight sums (this thread's key
// lane shares lp, reduced over the group), then the output: fp16 / bfloat16
// rows when the unit is one piece, else the unnormalised O rows and (m, l) --
// staged in shared memory for a cluster merge, or written to the workspace
// slot of the piece. o[h][k] is output dim 128 h + key of row 8 g + k.
template <class T>
__device__ __forceinline__ void tc_write_piece(const DecodeParams& p, const Piece& pc, const float (&o)[T::kSlabs][8],
                                               const float (&lp)[8], uint8_t* smem, float* rf, float* red, int g,
                                               int warp, int lane, int key) {
  constexpr int D = T::D, S = T::kSlabs, NR = T::kGroupRows;
  const int rb = NR * g, bid = 1 + g;
  {
    float v[NR];
#pragma unroll
    for (int r = 0; r < NR; ++r) v[r] = lp[r];
    const float sum = warp_transpose_reduce<false, NR>(v, lane);
    if (lane < NR) red[(warp & 3) * NR + lane] = sum;
  }
  named_bar_sync(bid, 128);
  if ((warp & 3) == 0 && lane < NR)
    rf[kRowL * 32 + rb + lane] = (red[lane] + red[NR + lane]) + (red[2 * NR + lane] + red[3 * NR + lane]);
  named_bar_sync(bid, 128);
  const bool direct = pc.npieces == 1;
#pragma unroll
  for (int k = 0; k < NR; ++k) {
    const int r = rb + k;
    if (r >= pc.R) break;
    const float L = rf[kRowL * 32 + r];
    if (direct) {
      const int i = r / p.G, hl = r % p.G;
      __half* dst = p.out + (static_cast<long long>(pc.q0 + i) * p.Hq + pc.kh * p.G + hl) * D;
      const float inv = L > 0.f ? p.out_scale / L : 0.f;
#pragma unroll
      for (int h = 0; h < S; ++h)
        reinterpret_cast<uint16_t*>(dst)[128 * h + key] = pack1<T::QB>(o[h][k] * inv);
    } else if (p.cluster > 1) {
      float* dst = reinterpret_cast<float*>(smem) + r * D;  // the staged rows, over the K ring
#pragma unroll
      for (int h = 0; h < S; ++h) dst[128 * h + key] = o[h][k];
    } else {
      float* dst = p.ws_o + (static_cast<long long>(pc.slot) * p.rows_padded + r) * D;
#pragma unroll
      for (int h = 0; h < S; ++h) __stcg(dst + 128 * h + key, o[h][k]);
    }
  }
  if (!direct && key < NR && rb + key < pc.R) {
    const int r = rb + key;
    const float mu = rf[kRowMu * 32 + r];
    const float2 ml = make_float2(mu == -INFINITY ? -INFINITY : mu - T::kBias, rf[kRowL * 32 + r]);
    if (p.cluster > 1)
      reinterpret_cast<float2*>(smem + T::kOffStageMl)[r] = ml;
    else
      __stcg(reinterpret_cast<float2*>(p.ws_ml + (static_cast<long long>(pc.slot) * p.rows_padded + r) * 2), ml);
  }
}

// The softmax warps: NG warpgroups share the keys of a block -- thread i of a
// group owns TMEM lane i (key i of a block for S^T, output dims i and i + 128
// for O^T) -- and split the query rows: group g takes rows 8 g .. 8 g + 7,
// with their running maxima, sums and O^T columns, so the groups never wait on
// each other inside a block.
template <class T>
__device__ __forceinline__ void softmax_role(const DecodeParams& p, const int* s_pre, WorkIter& it, Piece& pc,
                                             uint8_t* smem, uint32_t sbase, uint32_t tmem, bool& ok) {
  constexpr int D = T::D, NBK = T::NBK, NBV = T::NBV, S = T::kSlabs, NR = T::kGroupRows;
  constexpr int NST = T::kSoftThreads;
  (void)NBK;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = warp >> 2;              // row group
  const int key = tid & 127;            // TMEM lane of this thread
  const int rb = NR * g;                // first row of this group
  float* rf = reinterpret_cast<float*>(smem + T::kOffRow);
  int* ri = reinterpret_cast<int*>(smem + T::kOffRow);
  float* red = reinterpret_cast<float*>(smem + T::kOffRed) + 4 * NR * g;  // [4 warps][8 rows]
  const uint32_t fullv0 = sbase + T::kOffBars + 16 * NBK, bx = fullv0 + 16 * NBV;
  auto bar = [&](int i) -> uint32_t { return bx + 8 * i; };
  const uint32_t tl = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);  // this warp's TMEM lanes
  const uint32_t qs = sbase + T::kOffQ, pt = sbase + T::kOffPt;
  uint32_t bq = 0;
  // A piece's q terms (the B operand of S^T: K-major, 128-byte swizzle, the
  // three terms stacked on N), row score factors and visible key limits; the
  // previous piece's S^T products are complete (its softmax read them all).
  // Item t < 256 (thread t, and t + 128 with a single group): row t / 8,
  // dims [(t % 8) D / 8, (t % 8 + 1) D / 8).
  auto q_setup = [&](const Piece& pq) {
    for (int item = tid; item < 256; item += NST) {
      const int r = item >> 3, part = item & 7;
      constexpr int NCH = D / 128;  // 16-dim chunks per thread
      const __half* qrow = nullptr;
      if (r < pq.R) {
        const int i = r / p.G, hl = r % p.G;
        qrow = p.q + (static_cast<long long>(pq.q0 + i) * p.Hq + pq.kh * p.G + hl) * D;
      }
      uint4 qv[NCH][2];
      float mx = 0.f;
#pragma unroll
      for (int c = 0; c < NCH; ++c) {
        const int d0 = part * (D / 8) + 16 * c;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          qv[c][hh] = qrow ? __ldg(reinterpret_cast<const uint4*>(qrow + d0 + 8 * hh)) : make_uint4(0u, 0u, 0u, 0u);
          const uint32_t w[4] = {qv[c][hh].x, qv[c][hh].y, qv[c][hh].z, qv[c][hh].w};
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const float2 f = pair_to_float2<T::QB>(w[k]);
            mx = fmaxf(mx, fmaxf(fabsf(f.x), fabsf(f.y)));
          }
        }
      }
#pragma unroll
      for (int o = 1; o < 8; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      // 2^e with the row's largest |q| * 2^e in [128, 256); for an fp16 q, e
      // lies in [-8, 31]; a bfloat16 q reaches further, and e is held to
      // [-126, 126] so that 2^e and 2^-e stay normal floats (only rows whose
      // largest |q| is below 2^-119 then keep fewer than 11 bits)
      const int e = mx > 0.f ? max(-126, min(126, 134 - static_cast<int>((__float_as_uint(mx) >> 23) & 255u)))
                             : 0;
      const float up = __uint_as_float(static_cast<uint32_t>(127 + e) << 23);
#pragma unroll
      for (int c = 0; c < NCH; ++c) {
        const int d0 = part * (D / 8) + 16 * c;
        uint32_t tw[3][4];
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const uint32_t w[4] = {qv[c][hh].x, qv[c][hh].y, qv[c][hh].z, qv[c][hh].w};
#pragma unroll
          for (int k = 0; k < 4; k += 2) {
            uint32_t a[3], b[3];
            const float2 fa = pair_to_float2<T::QB>(w[k]);
            const float2 fb = pair_to_float2<T::QB>(w[k + 1]);
            split3_e4m3(pack_half2(fa.x * up, fa.y * up), a[0], a[1], a[2]);
            split3_e4m3(pack_half2(fb.x * up, fb.y * up), b[0], b[1], b[2]);
#pragma unroll
            for (int t = 0; t < 3; ++t) tw[t][2 * hh + k / 2] = a[t] | (b[t] << 16);
          }
        }
        const uint32_t off = (d0 >> 7) * T::kQSlab + r * 128 + ((((d0 & 127) >> 4) ^ (r & 7)) << 4);
#pragma unroll
        for (int t = 0; t < 3; ++t)
          asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(qs + t * T::kN * 128 + off), "r"(tw[t][0]),
                       "r"(tw[t][1]), "r"(tw[t][2]), "r"(tw[t][3])
                       : "memory");
      }
      if (part == 0) {
        int lo = 0, hi = -1;
        if (r < pq.R) {
          hi = pq.L - pq.qlen + r / p.G;
          lo = p.window > 0 ? max(0, hi - p.window + 1) : 0;
        }
        rf[kRowFsl * 32 + r] = r < pq.R ? p.sl2 * __uint_as_float(static_cast<uint32_t>(127 - e) << 23) : 0.f;
        rf[kRowMu * 32 + r] = -INFINITY;
        ri[kRowLo * 32 + r] = lo;
        ri[kRowHi * 32 + r] = hi;
      }
    }
    fence_proxy_async_smem();
  };
  auto load8 = [&](const float* src, float (&dst)[NR]) {
#pragma unroll
    for (int k = 0; k < NR / 4; ++k) {
      const float4 f = reinterpret_cast<const float4*>(src)[k];
      dst[4 * k] = f.x; dst[4 * k + 1] = f.y; dst[4 * k + 2] = f.z; dst[4 * k + 3] = f.w;
    }
  };

  while (tc_next_piece<T>(p, s_pre, it, pc)) {
    const int nblk = (pc.ntiles + T::kBlkTiles - 1) / T::kBlkTiles;
    q_setup(pc);
    named_bar_sync(T::kBarAll, NST);
    if (tid == 0) mbar_arrive(bar(kBarQFull));
    float fs[NR];  // score factor of each row of this group
    load8(rf + kRowFsl * 32 + rb, fs);
    float lp[NR];  // this key lane's share of each row's weight sum
#pragma unroll
    for (int r = 0; r < NR; ++r) lp[r] = 0.f;

    for (int i = 0; i < nblk; ++i) {
      const uint32_t b = bq + i;
      const int sv = b % NBV, sb = b & 1;
      const int key0 = (pc.first_tile + T::kBlkTiles * i) * kTileKeys;
      const int nvalid = min(128, kTileKeys * (pc.ntiles - T::kBlkTiles * i));  // keys loaded
      // ---- this key's scores for the group's 8 rows (three term slices)
      float x[NR];
      if (ok) ok = mbar_wait(bar(kBarSFull + sb), (b >> 1) & 1, p.timeout_ns);
      ok = __all_sync(0xffffffffu, ok);  // tcgen05.ld is warp-collective
      tc_fence_after();
      if (ok) {
        float y[NR], z[NR];
        const uint32_t sc = tl + T::kColS + T::kNT * sb + rb;
        tmem_ld8(sc, x);
        tmem_ld8(sc + 32, y);
        tmem_ld8(sc + 64, z);
        tmem_wait_ld();
#pragma unroll
        for (int r = 0; r < NR; ++r) x[r] = (x[r] + y[r]) + z[r];
      } else {
#pragma unroll
        for (int r = 0; r < NR; ++r) x[r] = 0.f;
      }
      tc_fence_before();
      __syncwarp();
      if (ok && lane == 0) mbar_arrive(bar(kBarSEmpty + sb));
      tc_scale_mask<T>(x, fs, fs, key0, nvalid, pc, ri, rb, key);
      // ---- running maximum per row (see tc_raise_max)
      float mu[NR];
      const bool rescale = tc_raise_max<T>(x, mu, rf, ri, red, g, warp, lane);
      // ---- weights 2^(x - mu + kBias) (<= 2^8) and the row sums
#pragma unroll
      for (int r = 0; r < NR; ++r) x[r] = ex2(x[r] - (mu[r] == -INFINITY ? 0.f : mu[r] - T::kBias));
      if (rescale) {
#pragma unroll
        for (int r = 0; r < NR; ++r) lp[r] = lp[r] * rf[kRowAl * 32 + rb + r] + x[r];
      } else {
#pragma unroll
        for (int r = 0; r < NR; ++r) lp[r] += x[r];
      }
      // ---- the P.V operands are free once the previous block's product is done
      if (ok && b >= 1) ok = mbar_wait(bar(kBarPvDone), (b - 1) & 1, p.timeout_ns);
      ok = __all_sync(0xffffffffu, ok);
      tc_fence_after();
      if (rescale && i > 0 && ok) {
        // O^T columns of this group's rows whose running maximum was raised
#pragma unroll 1
        for (int c = 0; c < 3 * S; ++c) {
          float o[NR];
          tmem_ld8(tl + T::kColO + 32 * c + rb, o);
          tmem_wait_ld();
#pragma unroll
          for (int r = 0; r < NR; ++r) o[r] *= rf[kRowAl * 32 + rb + r];
          tmem_st8(tl + T::kColO + 32 * c + rb, o);
        }
        tmem_wait_st();
      }
      // ---- P^T, three e4m3 terms: this key's 8 row weights are the 8-byte
      // piece 8 g of a 32-byte row (k = key) of an MN-major operand in the
      // 32-byte swizzle layout (8-key atoms of 256 bytes; the 16-byte halves
      // swap in rows 4-7)
      {
        uint32_t tt[3][NR / 2];
#pragma unroll
        for (int k = 0; k < NR / 2; ++k)
          split3_e4m3(pack_half2(x[2 * k], x[2 * k + 1]), tt[0][k], tt[1][k], tt[2][k]);
        const uint32_t row = pt + (key >> 3) * 256 + (key & 7) * 32 +
                             ((((g >> 1) ^ ((key & 7) >> 2)) << 4) | ((g & 1) << 3));
#pragma unroll
        for (int t = 0; t < 3; ++t)
          asm volatile("st.shared.v2.b32 [%0], {%1,%2};" ::"r"(row + t * T::kPtTerm),
                       "r"(tt[t][0] | (tt[t][1] << 16)), "r"(tt[t][2] | (tt[t][3] << 16))
                       : "memory");
      }
      // ---- V rows of keys past the sequence end or not loaded (stale or
      // unwritten bytes, NaN codes included) are zeroed in the ring by the first
      // group: the P.V product reads V there, and a zero weight must not meet a NaN
      const int lim = min(nvalid, pc.L - key0);
      if (g == 0 && lim < 128) {
        if (ok) ok = mbar_wait(fullv0 + 8 * sv, (b / NBV) & 1, p.timeout_ns);
        ok = __all_sync(0xffffffffu, ok);
        if (ok && key >= lim) {
          const uint32_t vrow = sbase + T::kOffV + sv * T::kKBlk + key * 128;
#pragma unroll
          for (int sl = 0; sl < S; ++sl)
#pragma unroll
            for (int c = 0; c < 8; ++c)
              asm volatile("st.shared.v4.b32 [%0], {%1,%1,%1,%1};" ::"r"(vrow + sl * T::kSlabBlk + 16 * c), "r"(0u)
                           : "memory");
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (ok && lane == 0) mbar_arrive(bar(kBarPFull));
    }
    bq += nblk;

    // ---- epilogue: O^T (this thread: dims key, key + 128) of the group's
    // rows, row sums, output
    if (ok) ok = mbar_wait(bar(kBarPvDone), (bq - 1) & 1, p.timeout_ns);
    ok = __all_sync(0xffffffffu, ok);
    tc_fence_after();
    float o[S][NR];
#pragma unroll
    for (int h = 0; h < S; ++h) {
      if (ok) {
        float y[NR], z[NR];
        const uint32_t oc = tl + T::kColO + T::kNT * h + rb;
        tmem_ld8(oc, o[h]);
        tmem_ld8(oc + 32, y);
        tmem_ld8(oc + 64, z);
        tmem_wait_ld();
#pragma unroll
        for (int r = 0; r < NR; ++r) o[h][r] = (o[h][r] + y[r]) + z[r];
      } else {
#pragma unroll
        for (int r = 0; r < NR; ++r) o[h][r] = 0.f;
      }
    }
    tc_fence_before();
    tc_write_piece<T>(p, pc, o, lp, smem, rf, red, g, warp, lane, key);
    named_bar_sync(T::kBarAll, NST);  // the row state and red[] are rewritten by the next piece
  }
  if (!ok && lane == 0) raise_error(p.error_flag, kErrTimeout);
}

// Cluster merge of a fixed split (p.cluster = S pieces per unit, the S CTAs
// of one cluster, cluster rank = split index): every CTA has staged its
// partial (m, l) per row and its unnormalised O rows in its shared memory;
// CTA s merges the float4 groups g of the unit's rows with g % S == s, reading
// all S partials through distributed shared memory (all loads of an item in
// flight at once), and writes them as the split combine would: M = max m,
// w = 2^(m - M), out = sum w O / sum w l. A CTA that got no piece staged
// m = -inf (weight 0; its O rows are never written and are not used). A unit
// covered by one piece (or none) was written by its piece.
template <class T>
__device__ __forceinline__ void cluster_merge(const DecodeParams& p, uint32_t sbase) {
  constexpr int D = T::D, Q4 = D / 4, SMAX = kMaxCluster;
  const int S = p.cluster;
  const int rank = static_cast<int>(cluster_rank());
  const int u = blockIdx.x / S;
  const int b = u / p.hgn, kh = (u % p.hgn) * p.hg;
  int L, t0, n, q0, qn;
  seq_span(p, b, false, L, t0, n, q0, qn);
  if (n == 0) return;
  const int chunk = (n + S - 1) / S;
  if ((n + chunk - 1) / chunk <= 1) return;
  const int R = p.G * qn;
  uint32_t peer[SMAX];  // each peer's shared memory base in the cluster window
#pragma unroll
  for (int s = 0; s < SMAX; ++s) peer[s] = s < S ? peer_smem(sbase, s) : 0u;
  for (int item = rank + S * static_cast<int>(threadIdx.x); item < R * Q4; item += S * T::kThreads) {
    const int r = item / Q4, c4 = item % Q4;
    float2 ml[SMAX];
    float4 o[SMAX];
#pragma unroll
    for (int s = 0; s < SMAX; ++s) {
      if (s < S) {
        ml[s] = ld_peer_f2(peer[s] + T::kOffStageMl + 8 * r);
        o[s] = ld_peer_f4(peer[s] + (r * D + 4 * c4) * 4);
      }
    }
    float M = -INFINITY;
#pragma unroll
    for (int s = 0; s < SMAX; ++s)
      if (s < S) M = fmaxf(M, ml[s].x);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float lsum = 0.f;
#pragma unroll
    for (int s = 0; s < SMAX; ++s) {
      if (s < S && ml[s].x != -INFINITY) {  // an empty piece staged nothing
        const float w = ex2(ml[s].x - M);
        lsum += w * ml[s].y;
        acc.x += w * o[s].x; acc.y += w * o[s].y; acc.z += w * o[s].z; acc.w += w * o[s].w;
      }
    }
    const float inv = lsum > 0.f ? p.out_scale / lsum : 0.f;
    const int i = r / p.G, hl = r % p.G;
    uint16_t* dst = reinterpret_cast<uint16_t*>(p.out) +
                    (static_cast<long long>(q0 + i) * p.Hq + kh * p.G + hl) * D + 4 * c4;
    const uint32_t lo = pack2<T::QB>(acc.x * inv, acc.y * inv), hi = pack2<T::QB>(acc.z * inv, acc.w * inv);
    *reinterpret_cast<uint2*>(dst) = make_uint2(lo, hi);
  }
}

// The producer warps (kProducerWarp: K ring, the next warp: V ring): each
// TMA-loads the rows of its operand for every block of its CTA's pieces, all
// boxes of a block at once (lane l: tile l / kSlabs of the block, 128-byte
// slab l % kSlabs), and waits only for its own ring's empty stages, so K runs
// ahead of V. Block table entries are read 32 tiles (4 blocks) at a time, the
// next group in flight. Rings and their barriers: K stages at offset 0, V
// stages at kOffV; fullK[NBK], emptyK[NBK], fullV[NBV], emptyV[NBV] first in
// the barrier area.
template <class T>
__device__ __forceinline__ void tc_producer_role(const DecodeParams& p, const int* s_pre, WorkIter& it, Piece& pc,
                                                 const CUtensorMap* tm_k, const CUtensorMap* tm_v, uint32_t sbase,
                                                 bool& ok) {
  constexpr int NBK = T::NBK, NBV = T::NBV;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t fullk0 = sbase + T::kOffBars, emptyk0 = fullk0 + 8 * NBK;
  const uint32_t fullv0 = emptyk0 + 8 * NBK, emptyv0 = fullv0 + 8 * NBV;
  const bool is_v = warp != T::kProducerWarp;
  const int nb = is_v ? NBV : NBK;
  const uint32_t fullb = is_v ? fullv0 : fullk0, emptyb = is_v ? emptyv0 : emptyk0;
  const uint32_t ringb = sbase + (is_v ? T::kOffV : 0);
  const CUtensorMap* tm = is_v ? tm_v : tm_k;
  const uint64_t pol = l2_policy_evict_first();
  uint32_t bq = 0, posted = 0;  // blocks walked; blocks whose loads were all issued
  while (work_next(p, s_pre, it, pc)) {
    if (pc.ntiles == 0) continue;
    const int nblk = (pc.ntiles + T::kBlkTiles - 1) / T::kBlkTiles;
    const int32_t* row = p.block_table + static_cast<long long>(pc.b) * p.max_blocks;
    auto load_group = [&](int t) -> int {
      int blk = 0;
      if (t + lane < pc.ntiles) blk = __ldg(row + (pc.first_tile + t + lane) / p.tiles_per_block);
      return blk;
    };
    // block table entries 32 tiles (4 blocks) at a time, the next group in flight
    int cur = load_group(0), nxt = pc.ntiles > 32 ? load_group(32) : 0;
    for (int i = 0; i < nblk; ++i) {
      const int t0 = i * T::kBlkTiles;
      if (t0 > 0 && t0 % 32 == 0) {
        cur = nxt;
        nxt = t0 + 32 < pc.ntiles ? load_group(t0 + 32) : 0;
      }
      const uint32_t b = bq + i;
      const int st = b % nb;
      const int ntb = min(T::kBlkTiles, pc.ntiles - t0);
      if (lane == 0) {
        if (ok && b >= static_cast<uint32_t>(nb)) ok = mbar_wait(emptyb + 8 * st, ((b / nb) - 1) & 1, p.timeout_ns);
        if (ok && p.inject == 1) ok = false;  // injected fault: the rings stay empty
        if (ok) {
          mbar_arrive_expect_tx(fullb + 8 * st, ntb * T::kSlabs * T::kTileBox);
          posted = b + 1;
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      // lane l: tile l / kSlabs of the block, slab l % kSlabs (all boxes at once)
      const int j = min(lane / T::kSlabs, T::kBlkTiles - 1);
      int blk = __shfl_sync(0xffffffffu, cur, (t0 % 32) + j);
      if (!ok) continue;
      if (lane < T::kSlabs * ntb) {
        if (blk < 0 || blk >= p.num_blocks) {
          if (!is_v) raise_error(p.error_flag, kErrBlockId);
          blk = 0;
        }
        const int gt = pc.first_tile + t0 + j;
        const int z = blk * p.block_size + (gt % p.tiles_per_block) * kTileKeys;
        const int sl = lane % T::kSlabs;
        tma_load_3d(ringb + st * T::kKBlk + sl * T::kSlabBlk + j * T::kTileBox, tm, fullb + 8 * st, sl * 128,
                    pc.kh, z, pol);
      }
    }
    bq += nblk;
  }
  if (lane == 0) {
    if (!ok) raise_error(p.error_flag, kErrTimeout);
    // every load issued lands before the CTA exits: a block's loads are all
    // issued once its transaction count is posted
    for (uint32_t k = posted > static_cast<uint32_t>(nb) ? posted - nb : 0; k < posted; ++k)
      if (!mbar_wait(fullb + 8 * (k % nb), (k / nb) & 1, kDrainLimitNs)) break;
  }
}

template <class T>
__global__ void __launch_bounds__(T::kThreads, 1)
    decode_tc8_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                      const DecodeParams p) {
  constexpr int D = T::D, NBK = T::NBK, NBV = T::NBV, KS = D / 32;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t fullk0 = sbase + T::kOffBars, emptyk0 = fullk0 + 8 * NBK;
  const uint32_t fullv0 = emptyk0 + 8 * NBK, emptyv0 = fullv0 + 8 * NBV, bx = emptyv0 + 8 * NBV;
  auto bar = [&](int i) -> uint32_t { return bx + 8 * i; };
  int* s_pre = reinterpret_cast<int*>(smem + T::kOffPre);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + T::kOffTmem);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < NBK; ++s) {
      mbar_init(fullk0 + 8 * s, 1);
      mbar_init(emptyk0 + 8 * s, 1);  // the S^T commit
    }
    for (int s = 0; s < NBV; ++s) {
      mbar_init(fullv0 + 8 * s, 1);
      mbar_init(emptyv0 + 8 * s, 1);  // the P.V commit
    }
    mbar_init(bar(kBarSFull), 1);
    mbar_init(bar(kBarSFull + 1), 1);
    mbar_init(bar(kBarSEmpty), 4 * T::NG);  // the softmax warps
    mbar_init(bar(kBarSEmpty + 1), 4 * T::NG);
    mbar_init(bar(kBarPFull), 4 * T::NG);
    mbar_init(bar(kBarPvDone), 1);
    mbar_init(bar(kBarQFull), 1);
    mbar_init(bar(kBarFinal), 1);
    fence_mbar_init();
  }
  if (warp == T::kMmaWarp) {
    tmem_alloc(smem_u32(tmem_slot), T::kTmemCols);
    tmem_relinquish();
  }
  if (warp == T::kProducerWarp && lane == 0) {
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
  }
  // P^T starts as zeros: the columns of rows no group owns (a unit of fewer
  // than four row tiles) are multiplied but never written or read
  for (int i = threadIdx.x; i < 3 * T::kPtTerm / 16; i += T::kThreads)
    asm volatile("st.shared.v4.b32 [%0], {%1,%1,%1,%1};" ::"r"(sbase + T::kOffPt + 16 * i), "r"(0u) : "memory");
  fence_proxy_async_smem();
  // a CTA of a cluster that gets no piece (a unit with fewer tiles than
  // pieces) contributes nothing to the merge
  if (threadIdx.x < 32)
    reinterpret_cast<float2*>(smem + T::kOffStageMl)[threadIdx.x] = make_float2(-INFINITY, 0.f);
  // programmatic dependent launch: no global memory was touched above
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (p.num_splits == 0 && warp == 0) balanced_prefix(p, s_pre, lane);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  WorkIter it;
  work_init(p, s_pre, it);
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  Piece pc;
  bool ok = true;

  if (warp == T::kProducerWarp || warp == T::kProducerWarp + 1) {
    tc_producer_role<T>(p, s_pre, it, pc, &tm_k, &tm_v, sbase, ok);
  } else if (warp == T::kMmaWarp) {
    // ------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      uint32_t bq = 0, pq = 0;
      bool any = false;
      const uint32_t qb = sbase + T::kOffQ, pt = sbase + T::kOffPt;
      while (work_next(p, s_pre, it, pc)) {
        if (pc.ntiles == 0) continue;
        const int nblk = (pc.ntiles + T::kBlkTiles - 1) / T::kBlkTiles;
        if (ok) ok = mbar_wait(bar(kBarQFull), pq & 1, p.timeout_ns);
        ++pq;
        tc_fence_after();
        for (int i = 0; i <= nblk; ++i) {
          if (i < nblk) {  // S^T of block i
            const uint32_t b = bq + i;
            const int sk = b % NBK, sb = b & 1;
            if (ok) ok = mbar_wait(fullk0 + 8 * sk, (b / NBK) & 1, p.timeout_ns);
            if (ok && b >= 2) ok = mbar_wait(bar(kBarSEmpty + sb), ((b >> 1) - 1) & 1, p.timeout_ns);
            tc_fence_after();
            if (ok) {
              const uint32_t kbase = sbase + sk * T::kKBlk;
#pragma unroll
              for (int ks = 0; ks < KS; ++ks) {
                const uint32_t koff = (ks >> 2) * T::kSlabBlk + (ks & 3) * 32;
                const uint32_t qoff = (ks >> 2) * T::kQSlab + (ks & 3) * 32;
                mma_e4m3(tmem + T::kColS + T::kNT * sb, sdesc_sw128(kbase + koff), sdesc_sw128(qb + qoff),
                         T::kIdescS, ks != 0);
              }
              mma_commit(bar(kBarSFull + sb));
              mma_commit(emptyk0 + 8 * sk);
              any = true;
            }
          }
          if (i >= 1) {  // O^T += V^T P^T of block i - 1, V^T read in place (MN-major)
            const uint32_t b = bq + i - 1;
            const int sv = b % NBV;
            if (ok) ok = mbar_wait(fullv0 + 8 * sv, (b / NBV) & 1, p.timeout_ns);
            if (ok) ok = mbar_wait(bar(kBarPFull), b & 1, p.timeout_ns);
            tc_fence_after();
            if (ok) {
              const uint32_t vbase = sbase + T::kOffV + sv * T::kKBlk;
#pragma unroll
              for (int h = 0; h < T::kSlabs; ++h)
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                  mma_e4m3(tmem + T::kColO + T::kNT * h, sdesc_sw128_mn(vbase + h * T::kSlabBlk + kk * 4096),
                           sdesc_sw32_mn(pt + kk * 1024, T::kPtTerm), T::kIdescO, (i > 1 || kk > 0) ? 1u : 0u);
              mma_commit(bar(kBarPvDone));
              mma_commit(emptyv0 + 8 * sv);
              any = true;
            }
          }
        }
        bq += nblk;
      }
      if (!ok) raise_error(p.error_flag, kErrTimeout);
      // every issued product completes before the tensor memory is freed
      if (any) {
        mma_commit(bar(kBarFinal));
        mbar_wait(bar(kBarFinal), 0, kDrainLimitNs);
      }
    }
    __syncwarp();
  } else {
    // ----------------------------------------------------------- softmax warps
    softmax_role<T>(p, s_pre, it, pc, smem, sbase, tmem, ok);
  }
  tc_fence_before();
  __syncthreads();
  if (p.cluster > 1) {
    cluster_sync();  // every CTA of the cluster has staged its partial
    cluster_merge<T>(p, sbase);
    cluster_sync();  // no CTA leaves while a peer still reads its shared memory
  }
  if (warp == T::kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, T::kTmemCols);
  }
}

// Host launch of the e4m3 tensor-core decode (one CTA per SM), with
// programmatic dependent launch and, for a cluster-merged fixed split,
// clusters of p.cluster CTAs; sets the shared-memory opt-in once per context.
template <class T>
cudaError_t launch_tc8(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeParams& p, int grid,
                       cudaStream_t stream) {
  static unsigned long long attr_ctx[64] = {};
  const cudaError_t e = once_per_context(attr_ctx, [] {
    return set_kernel_attributes(decode_tc8_kernel<T>, T::kSmemBytes);
  });
  if (e != cudaSuccess) return e;
  return launch_pdl(decode_tc8_kernel<T>, grid, T::kThreads, T::kSmemBytes, stream, p.cluster, tk, tv, p);
}

template <class T>
bool shape_tc8(int nt, KernelShape* out) {
  out->threads = T::kThreads;
  out->smem_bytes = T::kSmemBytes;
  out->rows_padded = 8 * nt;
  out->ctas_per_sm = 1;
  out->heads = 1;
  out->unit_cost = T::kUnitCost;
  out->fixed_pieces = 1;
  static unsigned long long ctx_done[64] = {};
  static int cache[64][kMaxCluster + 1] = {};
  max_active_clusters(decode_tc8_kernel<T>, T::kThreads, T::kSmemBytes, ctx_done, cache, out->max_clusters);
  return true;
}

}  // namespace pd
