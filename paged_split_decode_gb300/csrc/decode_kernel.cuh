// decode_kernel.cuh -- paged split-K decode attention for sm_103a.
//
// Computes, for every sequence b, query token i and query head h, the softmax
// of scale * q . k over the keys the token sees, weighted over V (the per-head
// paged decode of opengfx1030/vllm-rdna pull request #33, "Purpose"), reading
// K and V through an int32 block table from caches laid out
// [num_blocks, block_size, Hkv, D].
//
// GB300 design (the pull request's RDNA2 schedule is prior art only):
//  * Work unit = (sequence b, group of HG consecutive KV heads). All G*qlen
//    query rows of every head in the group are packed into one CTA, so each
//    K/V byte crosses HBM once. A tile is 16 keys of the HG heads: with HG > 1
//    one TMA box reads HG*128 contiguous bytes per key, which is what lets the
//    HBM stream run near the copy rate (one head per tile reads 256-512 B at
//    an Hkv-fold stride and tops out lower).
//  * Persistent grid (one or two CTAs per SM). The visible key tiles of all
//    units are laid end to end and cut into equal contiguous ranges, one per
//    CTA (balanced split-K). A fixed num_splits instead cuts each unit into
//    num_splits chunks handed out round robin.
//  * One producer warp walks the CTA's tiles, reads block-table entries 32 at
//    a time (the next group is prefetched while the current one is issued)
//    and issues TMA bulk-tensor loads of the K and V tiles into an NS-stage
//    ring of 128B-swizzled shared-memory slabs, completed on mbarriers.
//  * Consumer warps are (tile head th, key group kg, row group, D part): per
//    tile a warp forms S^T = K Q^T with mma.sync m16n8k16 (keys on M, query
//    rows on N, Q held in registers), masks, runs the online softmax with warp
//    shuffles, turns P into the B operand with movmatrix and accumulates
//    O^T = V^T P^T. fp8 e4m3 tiles are widened to fp16 in registers
//    (cvt.f16x2.e4m3x2), int8 tiles by an exact magic-number conversion; the K
//    scale is folded into the score scale and the V scale into the output.
//  * At the end of a unit piece the key groups of a head merge (m, l, O)
//    through shared memory (or, with one key group per head, each warp writes
//    its rows from registers). A unit covered by one piece is normalised and
//    written as fp16; otherwise the piece writes an fp32 partial and the
//    split-combine kernel, launched behind this one with programmatic
//    dependent launch, merges every split unit's partials in a fixed order.
//  * Every mbarrier wait is bounded in wall time; on expiry the kernel raises
//    an error bit and runs the rest of its control flow without waiting, so
//    named barriers stay consistent and the CTA always exits.
#pragma once
#include <cuda.h>
#include <cstdint>

#include "ptx.cuh"

namespace pd {

constexpr int kTileKeys = 16;      // keys per pipeline tile
constexpr int kMaxAutoB = 1024;    // sequences handled by the balanced split
// Split units are merged by a second kernel, which derives each unit's pieces
// and their workspace slots from the sequence lengths exactly as the decode
// kernel's walk cuts them (unit_layout below).
constexpr uint32_t kErrBlockId = 1u, kErrSeqLen = 2u, kErrTimeout = 4u, kErrQueryStart = 16u;
// Limit of the producer's final drain: every load it issued lands before the
// CTA exits, whatever the (possibly short) pipeline wait limit.
constexpr unsigned long long kDrainLimitNs = 2000000000ull;
constexpr float kLog2e = 1.4426950408889634f;

struct DecodeParams {
  const __half* q;            // [total_q, Hq, D] fp16 (bfloat16 bits for bfloat16 caches)
  __half* out;                // [total_q, Hq, D] same type as q
  const int32_t* block_table; // [B, max_blocks]
  const int32_t* seq_lens;    // [B]
  const int32_t* q_start;     // [B+1] query rows of each sequence; null: b*qlen, qlen each
  int total_q;                // rows of q and out
  float* ws_o;                // [slots, RP, D]   partial O (log2-domain weights)
  float* ws_ml;               // [slots, RP, 2]   partial (m, l), m in log2 units
  int n_merge;                // units the split combine visits (its grid's x extent; 0: no combine)
  int decode_grid;            // CTAs of the decode launch (the balanced split's cut)
  int rows_padded;            // RP: rows per partial slot
  uint32_t* error_flag;       // may be null
  int B, qlen, Hq, Hkv, G, R;  // qlen, R: the largest per sequence (R = G*qlen rows per head)
  int hg, hgn;                 // KV heads per tile; head groups per sequence (Hkv / hg)
  int rows_head;               // partial rows reserved per head of a unit (row tiles * 8)
  int max_blocks, block_size, num_blocks, tiles_per_block;
  int window;                 // <= 0: none
  int num_splits;             // 0: balanced
  int unit_cost;              // balanced: virtual tiles charged to the start of every unit
  float sl2;                  // scale * log2(e) * k_scale
  float out_scale;            // v_scale (1 for fp16)
  int out_bf16;               // q and out hold bfloat16 (bfloat16 caches)
  unsigned long long timeout_ns;  // limit of every pipeline wait
  int inject;                     // fault injection: 1 = the producer issues no load
  int cluster;                    // > 1: fixed split of this many pieces per unit, one CTA each, launched as
                                  // thread-block clusters that merge a unit's partials in shared memory
};

// KV element kinds: fp16, one byte per element (OCP e4m3fn or int8 codes), or
// bfloat16 (then q and out are bfloat16 too and the products run in bfloat16).
// The byte kinds also come with a bfloat16 q and out (kKvFp8Bq, kKvInt8Bq):
// the products still run in fp16 on the exactly widened codes, with each q row
// scaled by a power of two into fp16 (exact) and the factor taken back out of
// the row's scores.
constexpr int kKvF16 = 0, kKvFp8 = 1, kKvInt8 = 2, kKvBf16 = 3, kKvFp8Bq = 4, kKvInt8Bq = 5;

// The cache element kind of a kind, and whether q and out are bfloat16.
constexpr int cache_kind(int kv) { return kv == kKvFp8Bq ? kKvFp8 : kv == kKvInt8Bq ? kKvInt8 : kv; }
constexpr bool q_is_bf16(int kv) { return kv == kKvBf16 || kv == kKvFp8Bq || kv == kKvInt8Bq; }

// Row scale of a q row whose largest |value| is m (a float, >= 0): 2^e with
// m * 2^e in [2^14, 2^15) where that keeps 2^e and 2^-e normal floats, so the
// scaled bfloat16 values are exact fp16 values (8 significant bits, within
// fp16's range); e = 0 for an all-zero row.
__device__ __forceinline__ int q_row_exponent(float m) {
  if (!(m > 0.f)) return 0;
  const int eb = static_cast<int>((__float_as_uint(m) >> 23) & 255u);
  return max(-113, min(126, 141 - eb));
}
__device__ __forceinline__ float pow2f(int e) {  // 2^e for e in [-126, 127]
  return __uint_as_float(static_cast<uint32_t>(127 + e) << 23);
}

// Tensor-core product and output packing for the 16-bit operand type.
template <bool BF16>
__device__ __forceinline__ void mma_op(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                       uint32_t b1) {
  if constexpr (BF16) mma_16816_bf16(d, a, b0, b1);
  else mma_16816(d, a, b0, b1);
}
template <bool BF16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  if constexpr (BF16) return pack_bf162(lo, hi);
  else return pack_half2(lo, hi);
}
template <bool BF16>
__device__ __forceinline__ uint16_t pack1(float x) {
  return static_cast<uint16_t>(pack2<BF16>(x, 0.f) & 0xffffu);
}

// Two byte codes of `w` (its low or high 16 bits, byte 0 / 2 the lower index)
// widened to an fp16 pair, exactly. e4m3fn: the hardware conversion. int8:
// `w` must be pre-biased (w ^ 0x80808080, codes + 128 as unsigned bytes); each
// byte u is spliced under the fp16 exponent byte 0x64, giving 1024 + u exactly,
// and 1152 = 1024 + 128 is subtracted (the magic-number integer-to-float
// conversion; every value involved is an exactly representable integer).
template <int KV>
__device__ __forceinline__ uint32_t byte_pair_to_half2(uint32_t w, bool high) {
  if constexpr (KV == kKvFp8) {
    return e4m3x2_to_half2(static_cast<uint16_t>(high ? (w >> 16) : (w & 0xffffu)));
  } else {
    const uint32_t h = prmt(w, 0x64646464u, high ? 0x7362u : 0x5140u);
    const uint32_t bias = 0x64806480u;  // fp16 1152 in both halves
    __half2 r = __hsub2(*reinterpret_cast<const __half2*>(&h), *reinterpret_cast<const __half2*>(&bias));
    return *reinterpret_cast<uint32_t*>(&r);
  }
}
template <int KV>
__device__ __forceinline__ uint32_t byte_word_prep(uint32_t w) {
  if constexpr (KV == kKvInt8) return w ^ 0x80808080u;
  else return w;
}

template <int D_, int KV_, int NT_, int KG_, int NS_, int MINB_, int DS_ = (NT_ == 1 ? 1 : 2),
          int HG_ = 1, int RG_ = ((NT_ == 4 && DS_ == 2) ? 2 : 1)>
struct Cfg {
  static constexpr int D = D_, NT = NT_, KG = KG_, NS = NS_;
  // HG KV heads per tile: a tile is 16 keys of HG consecutive heads, which sit
  // next to each other in the cache; one TMA box per 128-byte slab covers all
  // HG heads (measured: boxes of one head each read the same bytes markedly
  // slower). The smem rows are (key, head) pairs, so the 16 rows of one head
  // meet only 8/HG of the eight 128B-swizzle phases: a 2- or 4-way bank
  // conflict on the consumers' reads, the smaller cost of the two. Each head
  // has its own consumer warps.
  static constexpr int HG = HG_;
  static constexpr int kMinBlocks = MINB_;              // resident CTAs per SM the plan targets
  static constexpr int KV = cache_kind(KV_);     // the cache's element kind
  static constexpr bool FP8 = KV == kKvFp8 || KV == kKvInt8;  // one-byte elements
  static constexpr bool BF16 = KV_ == kKvBf16;  // bfloat16 tensor-core operands
  static constexpr bool QB = q_is_bf16(KV_);     // q and out in bfloat16
  static constexpr bool kQScale = QB && !BF16;   // q rows scaled into fp16
  static constexpr int kElem = FP8 ? 1 : 2;
  static constexpr int kSlabElems = 128 / kElem;        // one 128-byte swizzle row
  static constexpr int kSlabs = D / kSlabElems;
  static constexpr int kSlabBytes = kTileKeys * HG * 128;  // [key][head][128 B], 1024-aligned
  static constexpr int kTileBytes = kSlabs * kSlabBytes;
  static constexpr int kStageBytes = 2 * kTileBytes;    // K tile then V tile
  // DS = 1: each consumer warp covers all of D for its 8-row tiles.
  // DS = 2 or 4: consumer warps come in groups splitting D into DS parts; each
  // warp of a group covers every row tile of its row group for its part of D,
  // widens only its part of a one-byte tile, and the group sums the partial
  // scores through shared memory in a fixed order (bitwise identical in every
  // warp of the group). RG row groups split a head's NT row tiles between
  // warps (NT == 4 with DS == 2: two groups of two, so a warp's fragments
  // fit; RG == NT: one row tile per warp, which keeps each warp's softmax to
  // its own rows at the price of every warp reading the whole tile).
  static constexpr int DS = DS_;
  static constexpr int RG = RG_;
  static_assert(NT % RG == 0, "row groups take equal shares of the row tiles");
  static constexpr int NTW = NT / RG;                    // row tiles per warp
  static constexpr int kConsumerWarps = HG * KG * RG * DS;
  static constexpr int kConsumerThreads = kConsumerWarps * 32;
  static constexpr int kThreads = kConsumerThreads + 32;
  static constexpr int RP = HG * NT * 8;                // partial rows per unit
  // Key groups merge through shared memory, which also stages the epilogue.
  // With one key group per head and several heads per tile, each warp's
  // (m, l, O) is final and is written straight from registers instead.
  static constexpr bool kSmemMerge = !(KG == 1 && HG > 1);
  static constexpr int kDP = D + 4;                     // merge row pitch (floats)
  static constexpr int kMergeOBytes = kSmemMerge ? HG * NT * 8 * kDP * 4 : 0;
  static constexpr int kMergeMLBytes = kSmemMerge ? HG * KG * NT * 8 * 2 * 4 : 0;
  static constexpr int kXchgFloats = 32 * 4 * NTW;       // one warp's partial S^T, lane-major
  static constexpr int kXchgBytes = DS > 1 ? HG * KG * RG * 2 * DS * kXchgFloats * 4 : 0;
  static_assert(HG == 1 || HG == 2 || HG == 4, "1, 2 or 4 heads per tile");
  // Key group kg takes the tiles whose ring sequence number is kg modulo KG
  // (across pieces, not within each). With NS a multiple of KG every use of a
  // stage belongs to the same key group, which consumes its tiles in order;
  // so when it waits on a stage's full barrier, the stage's previous phase is
  // its own, already consumed, and a parity wait can never be satisfied by a
  // phase two rounds old.
  static_assert(NS % KG == 0, "ring stages must be a multiple of the key groups");
  static_assert(HG * KG * RG <= 14, "named barriers 2.. cover every D group");
  static_assert(DS == 1 || DS == 2 || DS == 4, "D splits into 1, 2 or 4 parts");
  static_assert(!FP8 || (D / 16 / DS) % 4 == 0, "one-byte tiles need 64-dim parts");
  static constexpr int kOffMergeO = NS * kStageBytes;
  static constexpr int kOffMergeML = kOffMergeO + kMergeOBytes;
  static constexpr int kOffXchg = (kOffMergeML + kMergeMLBytes + 15) / 16 * 16;
  static constexpr int kOffBars = (kOffXchg + kXchgBytes + 15) / 16 * 16;
  static constexpr int kOffPre = kOffBars + 2 * NS * 8;
  static constexpr int kOffMisc = (kOffPre + (kMaxAutoB + 1) * 4 + 15) / 16 * 16;
  static constexpr int kSmemBytes = kOffMisc + 16 + 1024;  // + alignment slack
  static_assert(D % kSlabElems == 0, "D must be a multiple of the slab width");
  static_assert(D % 32 == 0, "D must be a multiple of 32");
};

// ---------------------------------------------------------------------------
// Work decomposition shared by the producer and the consumers. Both walk the
// same sequence of pieces, so the ring's tile order matches on both sides.
struct Piece {
  int b, kh, L;     // kh: first KV head of the unit's head group
  int first_tile;   // tile index (within the sequence) of the piece's first tile
  int ntiles;       // tiles in this piece (0: a zero-fill piece for an empty unit)
  int npieces;      // pieces the unit was cut into (1: write the output directly)
  int slot;         // workspace slot of this piece's partial (npieces > 1)
  int chunk;        // balanced mode: chunk the piece belongs to; fixed mode: split index
  int unit_t0;      // first visible tile of the unit (within the sequence)
  int unit;         // b * hgn + head group
  int first_slot_cta;  // balanced mode: the first chunk covering the unit
  long long unit_start;  // balanced mode: global index of the unit's first real tile
  int tile_lo_all;     // keys [tile_lo_all, tile_hi_all] are visible to every query
  int tile_hi_all;     // token of the unit (empty range when hi < lo)
  int qlen;            // query tokens of sequence b (0: nothing to compute or write)
  int R;               // G * qlen rows of the unit
  int q0;              // row of q / out holding the sequence's first query token
};

// Query tokens of sequence b: rows [q0, q0 + qn) of q and out. With
// per-sequence starts, a malformed range (decreasing, longer than qlen, or
// outside [0, total_q)) is reported and the sequence is skipped.
__device__ __forceinline__ void seq_queries(const DecodeParams& p, int b, bool report, int& q0,
                                            int& qn) {
  if (p.q_start == nullptr) {
    q0 = b * p.qlen;
    qn = p.qlen;
    return;
  }
  q0 = __ldg(p.q_start + b);
  qn = __ldg(p.q_start + b + 1) - q0;
  if (q0 < 0 || qn < 0 || qn > p.qlen || q0 > p.total_q - qn) {
    if (report && p.error_flag) atomicOr(p.error_flag, kErrQueryStart);
    q0 = 0;
    qn = 0;
  }
}

// Keys every query token of a sequence of length L sees: token 0 limits the
// top (position L - qlen), token qlen-1 the window's start.
__device__ __forceinline__ void common_range(const DecodeParams& p, int L, Piece& pc) {
  const int hi = L - pc.qlen;
  const int last = L - 1;
  int lo = 0;
  if (p.window > 0) lo = max(0, last - p.window + 1);
  pc.tile_lo_all = lo;
  pc.tile_hi_all = hi;
}

__device__ __forceinline__ void raise_error(uint32_t* flag, uint32_t bit) {
  if (flag) atomicOr(flag, bit);
}

// The visible tiles [t0, t0 + n) of a sequence of (validated) length L whose
// query rows are [q0, q0 + qn).
__device__ __forceinline__ void span_of(const DecodeParams& p, int L, int qn, int& t0, int& n) {
  if (L == 0 || qn == 0) { t0 = 0; n = 0; return; }
  int lo = 0;
  if (p.window > 0) {
    const int first = L - qn - p.window + 1;  // token 0's first visible key
    lo = first > 0 ? first : 0;
  }
  t0 = lo / kTileKeys;
  n = (L - 1) / kTileKeys - t0 + 1;
}

// Visible tile span of sequence b: tiles [t0, t0 + n), and its query rows
// [q0, q0 + qn). Validates seq_len and the query range.
__device__ __forceinline__ void seq_span(const DecodeParams& p, int b, bool report, int& L, int& t0,
                                         int& n, int& q0, int& qn) {
  L = p.seq_lens[b];
  const int cap = p.max_blocks * p.block_size;
  if (L < 0 || L > cap) {
    if (report) raise_error(p.error_flag, kErrSeqLen);
    L = L < 0 ? 0 : cap;
  }
  seq_queries(p, b, report, q0, qn);
  span_of(p, L, qn, t0, n);
}

// Balanced mode keeps, for batches of up to kSeqCacheB sequences, each
// sequence's validated (L, q0, qn) in the unused tail of the prefix array
// (read once from global memory while the prefix is formed), so that a CTA's
// walk over its pieces issues no dependent global load before its first
// block-table read.
constexpr int kSeqCacheB = 256;
constexpr int kCacheL = kSeqCacheB + 1, kCacheQ0 = 2 * kSeqCacheB + 1, kCacheQn = 3 * kSeqCacheB + 1;
static_assert(kCacheQn + kSeqCacheB <= kMaxAutoB + 1, "the cache fits in the prefix array");
__device__ __forceinline__ void seq_cache_put(const DecodeParams& p, int* s_pre, int b, int L, int q0, int qn) {
  if (p.B <= kSeqCacheB) {
    s_pre[kCacheL + b] = L;
    s_pre[kCacheQ0 + b] = q0;
    s_pre[kCacheQn + b] = qn;
  }
}
__device__ __forceinline__ void seq_span_cached(const DecodeParams& p, const int* s_pre, int b, int& L, int& t0,
                                                int& n, int& q0, int& qn) {
  if (p.B > kSeqCacheB) {
    seq_span(p, b, false, L, t0, n, q0, qn);
    return;
  }
  L = s_pre[kCacheL + b];
  q0 = s_pre[kCacheQ0 + b];
  qn = s_pre[kCacheQn + b];
  span_of(p, L, qn, t0, n);
}

// Balanced mode: the visible 16-key tiles of all units, laid end to end (T of
// them), are cut into Ce = min(grid, T) contiguous ranges of equal size (to
// one tile), one per CTA; chunk k is CTA k's range. A kernel whose pieces have
// a fixed cost (set-up, epilogue) charges unit_cost virtual tiles before the
// tiles of every unit, so a range that takes on a second unit gets fewer real
// tiles; a range's virtual tiles do no work. (A dynamic tail -- small
// chunks taken from a global counter -- was measured and lost: every chunk
// costs a key-group merge, a partial and a deeper combine tree.)
// start(k) = floor(T k / Ce) and owner(x) = max{k : start(k) <= x} =
// floor(((x + 1) Ce - 1) / T) in exact integer arithmetic, without 64-bit
// divisions (slow on the GPU, and on the path to a CTA's first load): with
// T = q Ce + r, floor(T k / Ce) = q k + floor(r k / Ce), and r k < Ce^2 fits
// 32 bits; owner starts from a single-precision estimate of x Ce / T and
// steps to the exact index along the monotone start().
struct ChunkPlan {
  long long T;
  int Ce;
  long long q;  // T / Ce
  int r;        // T % Ce
  __device__ __forceinline__ long long start(int k) const {
    return q * k + static_cast<long long>(static_cast<unsigned>(r) * static_cast<unsigned>(k) /
                                          static_cast<unsigned>(Ce));
  }
  __device__ __forceinline__ long long end(int k) const { return start(k + 1); }
  __device__ __forceinline__ int owner(long long x) const {
    int k = static_cast<int>(static_cast<float>(x) * (static_cast<float>(Ce) / static_cast<float>(T)));
    k = k < 0 ? 0 : (k > Ce - 1 ? Ce - 1 : k);
    while (k > 0 && start(k) > x) --k;
    while (k < Ce - 1 && start(k + 1) <= x) ++k;
    return k;
  }
};

__device__ __forceinline__ ChunkPlan make_chunk_plan(long long T, int grid) {
  ChunkPlan cp;
  cp.T = T;
  cp.Ce = T <= 0 ? 0 : static_cast<int>(T < grid ? T : grid);
  cp.q = cp.Ce > 0 ? T / cp.Ce : 0;
  cp.r = cp.Ce > 0 ? static_cast<int>(T - cp.q * cp.Ce) : 0;
  return cp;
}

// Balanced mode, warp 0: the prefix over sequences of their units' cost
// (visible tiles plus the per-unit charge, times the head groups), s_pre[b]
// for b = 0 .. B, and the per-sequence cache of lengths and query ranges.
__device__ __forceinline__ void balanced_prefix(const DecodeParams& p, int* s_pre, int lane) {
  int carry = 0;
  if (lane == 0) s_pre[0] = 0;
  for (int base = 0; base < p.B; base += 32) {
    const int b = base + lane;
    int v = 0;
    if (b < p.B) {
      int L, t0, n, q0, qn;
      seq_span(p, b, blockIdx.x == 0, L, t0, n, q0, qn);
      seq_cache_put(p, s_pre, b, L, q0, qn);
      v = n > 0 ? (n + p.unit_cost) * p.hgn : 0;
    }
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, v, o);
      if (lane >= o) v += y;
    }
    if (b < p.B) s_pre[b + 1] = carry + v;
    carry += __shfl_sync(0xffffffffu, v, 31);
  }
}

struct WorkIter {
  ChunkPlan cp;
  long long g, g_end, chunk_start;
  int chunk;        // the CTA's range (balanced mode)
  int b;
  int zero_b;       // next sequence to test for zero-fill, stepping by gridDim.x
  int zero_kh;      // head group of the next zero-fill piece
  long long piece;  // fixed-split mode
};

__device__ __forceinline__ void work_init(const DecodeParams& p, const int* s_pre, WorkIter& it) {
  const int c = blockIdx.x;
  if (p.num_splits == 0) {
    it.cp = make_chunk_plan(s_pre[p.B], gridDim.x);
    it.chunk = c;
    if (c < it.cp.Ce) {
      it.g = it.chunk_start = it.cp.start(c);
      it.g_end = it.cp.end(c);
    } else {
      it.g = it.g_end = it.chunk_start = 0;
    }
    // largest b with s_pre[b] <= g
    int lo = 0, hi = p.B - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s_pre[mid] <= it.g) lo = mid; else hi = mid - 1;
    }
    it.b = lo;
    it.zero_b = c;
    it.zero_kh = 0;
  } else {
    it.piece = c;
  }
}

// Produces the next piece; returns false when the CTA has no more work.
__device__ __forceinline__ bool work_next(const DecodeParams& p, const int* s_pre, WorkIter& it,
                                          Piece& pc) {
  const int C = gridDim.x;
  if (p.num_splits == 0) {
    while (it.g < it.g_end) {
      while (s_pre[it.b + 1] <= it.g) ++it.b;
      const int b = it.b;
      const int span = (s_pre[b + 1] - s_pre[b]) / p.hgn;  // unit_cost + visible tiles
      const long long off = it.g - s_pre[b];
      const int grp = static_cast<int>(off) / span;        // the prefix is int: off < 2^31
      const long long us = s_pre[b] + static_cast<long long>(grp) * span;
      const long long rs = us + p.unit_cost;  // the unit's first real tile
      const long long ue = us + span;
      if (it.g < rs) {  // the range starts in the unit's virtual tiles
        it.g = rs;
        if (it.g >= it.g_end) break;
      }
      const long long pe = ue < it.g_end ? ue : it.g_end;
      int L, t0, nn, q0, qn;
      seq_span_cached(p, s_pre, b, L, t0, nn, q0, qn);
      pc.b = b; pc.kh = grp * p.hg; pc.L = L; pc.unit_t0 = t0; pc.unit = b * p.hgn + grp;
      pc.qlen = qn; pc.R = p.G * qn; pc.q0 = q0;
      pc.first_tile = t0 + static_cast<int>(it.g - rs);
      pc.ntiles = static_cast<int>(pe - it.g);
      const int cf = it.cp.owner(rs), cl = it.cp.owner(ue - 1);
      pc.npieces = cl - cf + 1;
      pc.slot = 2 * it.chunk + (it.chunk_start < rs ? 1 : 0);
      pc.chunk = it.chunk;
      pc.first_slot_cta = cf;
      pc.unit_start = rs;
      common_range(p, L, pc);
      it.g = pe;
      return true;
    }
    // afterwards: zero rows of empty sequences b = c, c + C, ...
    while (it.zero_b < p.B) {
      const int b = it.zero_b;
      if (s_pre[b + 1] == s_pre[b]) {
        int q0, qn;
        seq_queries(p, b, false, q0, qn);
        pc.qlen = qn; pc.R = p.G * qn; pc.q0 = q0;
        pc.b = b; pc.kh = it.zero_kh * p.hg; pc.L = 0; pc.unit_t0 = 0;
        pc.unit = b * p.hgn + it.zero_kh;
        pc.first_tile = 0; pc.ntiles = 0; pc.npieces = 1; pc.slot = 0; pc.chunk = 0;
        pc.first_slot_cta = 0; pc.unit_start = 0;
        if (++it.zero_kh == p.hgn) { it.zero_kh = 0; it.zero_b += C; }
        return true;
      }
      it.zero_b += C;
    }
    return false;
  }
  const int S = p.num_splits;
  const long long total = static_cast<long long>(p.B) * p.hgn * S;
  while (it.piece < total) {
    const long long pi = it.piece;
    it.piece += C;
    const int u = static_cast<int>(pi / S), s = static_cast<int>(pi % S);
    const int b = u / p.hgn, kh = (u % p.hgn) * p.hg;
    int L, t0, n, q0, qn;
    seq_span(p, b, s == 0 && kh == 0, L, t0, n, q0, qn);
    pc.qlen = qn; pc.R = p.G * qn; pc.q0 = q0;
    const int chunk = (n + S - 1) / S;
    const int c0 = s * chunk;
    const int c1 = (c0 + chunk < n) ? c0 + chunk : n;
    if (n == 0) {
      if (s != 0) continue;
      pc.b = b; pc.kh = kh; pc.L = 0; pc.unit_t0 = 0; pc.unit = u;
      pc.first_tile = 0; pc.ntiles = 0; pc.npieces = 1; pc.slot = 0; pc.chunk = 0;
      pc.first_slot_cta = 0; pc.unit_start = 0;
      return true;
    }
    if (c0 >= c1) continue;
    pc.b = b; pc.kh = kh; pc.L = L; pc.unit_t0 = t0; pc.unit = u;
    pc.first_tile = t0 + c0;
    pc.ntiles = c1 - c0;
    pc.npieces = (n + chunk - 1) / chunk;
    pc.slot = u * S + s;
    pc.chunk = s;
    pc.first_slot_cta = 0; pc.unit_start = 0;
    common_range(p, L, pc);
    return true;
  }
  return false;
}

// Cluster merge of a fixed split whose S pieces per unit (p.cluster = S) are
// the S CTAs of one cluster (rank = split index). Every thread of the CTA
// calls it once, after the CTA's piece wrote its partial to the workspace
// (fp32 rows slot * RP + head * RH + r with slot = unit * S + split, O
// relative to m, m in log2 units): one cluster barrier (release / acquire at
// cluster scope, so every piece's partial is visible), then CTA s merges the
// float4 groups g of the unit's rows with g % S == s, reading the partials of
// the unit's pieces from L2 (all loads of an item in flight at once), and
// writes them as the split combine would: M = max m, w = 2^(m - M),
// out = sum w O / sum w l. A unit covered by one piece (or none) was written
// by its piece.
template <int D, int RP, int RH, int HG, int NTHREADS>
__device__ __forceinline__ void cluster_merge_ws(const DecodeParams& p) {
  constexpr int Q4 = D / 4, SMAX = 16;  // the largest cluster
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
  const int S = p.cluster;
  int rank;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(rank));
  const int u = blockIdx.x / S;
  const int b = u / p.hgn, kh = (u % p.hgn) * p.hg;
  int L, t0, n, q0, qn;
  seq_span(p, b, false, L, t0, n, q0, qn);
  if (n == 0) return;
  const int chunk = (n + S - 1) / S;
  const int np = (n + chunk - 1) / chunk;  // pieces that hold tiles (split indices 0 .. np - 1)
  if (np <= 1) return;
  const int R = p.G * qn;
  const long long slot0 = static_cast<long long>(u) * S;
  for (int item = rank + S * static_cast<int>(threadIdx.x); item < HG * R * Q4; item += S * NTHREADS) {
    const int hh = item / (R * Q4), rem = item - hh * (R * Q4);
    const int r = rem / Q4, c4 = rem % Q4;
    float2 ml[SMAX];
    float4 o[SMAX];
#pragma unroll
    for (int s = 0; s < SMAX; ++s) {
      if (s < np) {
        const long long prow = (slot0 + s) * RP + hh * RH + r;
        ml[s] = __ldcg(reinterpret_cast<const float2*>(p.ws_ml + prow * 2));
        o[s] = __ldcg(reinterpret_cast<const float4*>(p.ws_o + prow * D + 4 * c4));
      }
    }
    float M = -INFINITY;
#pragma unroll
    for (int s = 0; s < SMAX; ++s)
      if (s < np) M = fmaxf(M, ml[s].x);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float lsum = 0.f;
#pragma unroll
    for (int s = 0; s < SMAX; ++s) {
      if (s < np && ml[s].x != -INFINITY) {
        const float w = ex2(ml[s].x - M);
        lsum += w * ml[s].y;
        acc.x += w * o[s].x; acc.y += w * o[s].y; acc.z += w * o[s].z; acc.w += w * o[s].w;
      }
    }
    const float inv = lsum > 0.f ? p.out_scale / lsum : 0.f;
    const int i = r / p.G, hl = r % p.G;
    uint32_t* dst = reinterpret_cast<uint32_t*>(reinterpret_cast<uint16_t*>(p.out) +
                    (static_cast<long long>(q0 + i) * p.Hq + (kh + hh) * p.G + hl) * D + 4 * c4);
    if (p.out_bf16) {
      dst[0] = pack_bf162(acc.x * inv, acc.y * inv);
      dst[1] = pack_bf162(acc.z * inv, acc.w * inv);
    } else {
      dst[0] = pack_half2(acc.x * inv, acc.y * inv);
      dst[1] = pack_half2(acc.z * inv, acc.w * inv);
    }
  }
}

template <class Cfg>
__global__ void __launch_bounds__(Cfg::kThreads, Cfg::kMinBlocks)
    decode_paged_kernel(const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v, const DecodeParams p) {
  constexpr int D = Cfg::D, KG = Cfg::KG, NS = Cfg::NS;
  constexpr bool FP8 = Cfg::FP8, BF16 = Cfg::BF16;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  float* merge_o = reinterpret_cast<float*>(smem + Cfg::kOffMergeO);
  float* merge_ml = reinterpret_cast<float*>(smem + Cfg::kOffMergeML);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Cfg::kOffBars);  // full[NS], empty[NS]
  int* s_pre = reinterpret_cast<int*>(smem + Cfg::kOffPre);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool is_producer = warp == Cfg::kConsumerWarps;
  const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + NS);

  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, Cfg::HG * Cfg::RG * Cfg::DS);  // the warps of one key group
    }
    fence_mbar_init();
  }
  if (is_producer && lane == 0) {
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
  }
  // Launched with programmatic dependent launch: everything above touches no
  // global memory; wait here until the preceding grid in the stream has
  // completed and its writes are visible (a no-op without one).
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // Balanced mode: prefix over sequences of Hkv * (visible tiles), by warp 0.
  if (p.num_splits == 0 && warp == 0) balanced_prefix(p, s_pre, lane);
  __syncthreads();

  WorkIter it;
  work_init(p, s_pre, it);
  // the split-combine kernel may be scheduled now; it waits for this grid
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  Piece pc;

  if (is_producer) {
    // ------------------------------------------------------------ producer
    const uint64_t pol = l2_policy_evict_first();
    uint32_t q = 0, issued = 0;
    bool ok = true;
    while (work_next(p, s_pre, it, pc)) {
      if (pc.ntiles == 0) continue;
      const int32_t* row = p.block_table + static_cast<long long>(pc.b) * p.max_blocks;
      auto load_group = [&](int t) -> int {
        // lane i: physical block of tile t + i of this piece (0 past its end).
        // Validated where it is used, so the load stays in flight meanwhile.
        int blk = 0;
        if (t + lane < pc.ntiles) {
          const int tile = pc.first_tile + t + lane;
          blk = __ldg(row + tile / p.tiles_per_block);
        }
        return blk;
      };
      int cur = load_group(0);
      for (int t = 0; t < pc.ntiles; t += 32) {
        const int nxt = (t + 32 < pc.ntiles) ? load_group(t + 32) : -1;
        const int n = min(32, pc.ntiles - t);
        for (int i = 0; i < n; ++i, ++q) {
          int blk = __shfl_sync(0xffffffffu, cur, i);
          if (blk < 0 || blk >= p.num_blocks) {
            if (lane == 0) raise_error(p.error_flag, kErrBlockId);
            blk = 0;
          }
          const int stage = q % NS;
          const uint32_t fb = full0 + 8 * stage;
          if (lane == 0) {
            if (ok && q >= NS) ok = mbar_wait(empty0 + 8 * stage, ((q / NS) - 1) & 1, p.timeout_ns);
            if (ok && p.inject == 1) ok = false;  // injected fault: the ring stays empty
            if (ok) mbar_arrive_expect_tx(fb, Cfg::kStageBytes);
          }
          ok = __shfl_sync(0xffffffffu, ok, 0);
          if (!ok) continue;
          // lanes 0..kSlabs-1 load the K slabs, the next kSlabs lanes the V
          // slabs; one box covers 16 keys x HG heads x 128 bytes
          if (lane < 2 * Cfg::kSlabs) {
            const int tile = pc.first_tile + t + i;
            const int z = blk * p.block_size + (tile % p.tiles_per_block) * kTileKeys;
            const int sl = lane % Cfg::kSlabs;
            const bool is_v = lane >= Cfg::kSlabs;
            const uint32_t dst = smem_u32(smem + stage * Cfg::kStageBytes) +
                                 (is_v ? Cfg::kTileBytes : 0) + sl * Cfg::kSlabBytes;
            tma_load_3d(dst, is_v ? &tm_v : &tm_k, fb, sl * Cfg::kSlabElems, pc.kh, z, pol);
          }
          issued = q + 1;
        }
        cur = nxt;
      }
    }
    if (lane == 0) {
      if (!ok) raise_error(p.error_flag, kErrTimeout);
      // Drain: every issued load must land before the CTA's shared memory is
      // released. Loads past the consumers' last wait are none in a normal
      // run; after a timeout, wait (bounded) for whatever is still in flight.
      const uint32_t first = issued > NS ? issued - NS : 0;
      for (uint32_t k = first; k < issued; ++k) {
        if (!mbar_wait(full0 + 8 * (k % NS), (k / NS) & 1, kDrainLimitNs)) break;
      }
    }
    __syncwarp();
    if (p.cluster > 1) cluster_merge_ws<D, Cfg::RP, Cfg::NT * 8, Cfg::HG, Cfg::kThreads>(p);
    return;
  }

  // -------------------------------------------------------------- consumers
  constexpr int DS = Cfg::DS, NTW = Cfg::NTW, RG = Cfg::RG, HG = Cfg::HG;
  const int dh = warp % DS;                   // part of D
  const int rg = (warp / DS) % RG;            // row group: row tiles rg*NTW .. rg*NTW+NTW-1
  const int kg = (warp / (DS * RG)) % KG;     // key group
  const int th = warp / (DS * RG * KG);       // head of the tile (KV head pc.kh + th)
  const int pair = (th * KG + kg) * RG + rg;  // the D group this warp belongs to
  const int g = lane >> 2, t4 = lane & 3;
  constexpr int KSTEPS = D / 16;
  constexpr int KSW = KSTEPS / DS;             // k-steps of this warp's part of D
  constexpr int MTW = D / 16 / DS;             // m-tiles (16 output dims) of this warp
  float* xchg = reinterpret_cast<float*>(smem + Cfg::kOffXchg);
  uint32_t qf[KSW][NTW][2];
  float o[MTW][NTW][4];
  uint32_t q = 0;      // ring sequence number of the piece's first tile
  bool ok = true;

  while (work_next(p, s_pre, it, pc)) {
    // ---- per-piece setup: Q fragments (B operand) and per-row visible key limits
    // bfloat16 q over byte caches: each row's exponent from its largest |q|
    // over all of D (a warp that holds only part of D loads its rows whole,
    // all at once, so the warps sharing a row agree); each lane keeps the
    // exponent of row g (its q fragments) and the score factors of rows 2t4,
    // 2t4 + 1 (lane = 4 g + t4)
    int eq[NTW];          // exponent of q row g of row tile n
    float sl2r[NTW][2];   // score factor of rows 2t4 + c: p.sl2 / 2^e
#pragma unroll
    for (int n = 0; n < NTW; ++n) {
      eq[n] = 0;
      sl2r[n][0] = sl2r[n][1] = p.sl2;
    }
    if constexpr (Cfg::kQScale && DS > 1) {
      constexpr int W = D / 64;  // 32-bit words (bfloat16 pairs) per lane and row
      uint32_t wv[NTW * 8][W];
#pragma unroll
      for (int rr = 0; rr < NTW * 8; ++rr) {
        const int r = (rg * NTW + rr / 8) * 8 + rr % 8;
#pragma unroll
        for (int k = 0; k < W; ++k) wv[rr][k] = 0u;
        if (r < pc.R && pc.ntiles > 0) {
          const int i = r / p.G, hl = r % p.G;
          const uint32_t* row = reinterpret_cast<const uint32_t*>(
              p.q + (static_cast<long long>(pc.q0 + i) * p.Hq + (pc.kh + th) * p.G + hl) * D);
#pragma unroll
          for (int k = 0; k < W; ++k) wv[rr][k] = __ldg(row + W * lane + k);
        }
      }
#pragma unroll
      for (int rr = 0; rr < NTW * 8; ++rr) {
        float m = 0.f;
#pragma unroll
        for (int k = 0; k < W; ++k)
          m = fmaxf(m, fmaxf(fabsf(__uint_as_float(wv[rr][k] << 16)), fabsf(__uint_as_float(wv[rr][k] & 0xffff0000u))));
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        const int e = q_row_exponent(m), n = rr / 8, j = rr % 8;
        if (g == j) eq[n] = e;
        if (2 * t4 == j) sl2r[n][0] = p.sl2 * pow2f(-e);
        if (2 * t4 + 1 == j) sl2r[n][1] = p.sl2 * pow2f(-e);
      }
    }
#pragma unroll
    for (int n = 0; n < NTW; ++n) {
      const int r = (rg * NTW + n) * 8 + g;
      const __half* qrow = nullptr;
      if (r < pc.R && pc.ntiles > 0) {
        const int i = r / p.G, hl = r % p.G;
        qrow = p.q + (static_cast<long long>(pc.q0 + i) * p.Hq + (pc.kh + th) * p.G + hl) * D;
      }
#pragma unroll
      for (int ksl = 0; ksl < KSW; ++ksl) {
        const int ks = dh * KSW + ksl;
        int d0, d1;
        if constexpr (FP8) {
          // k-step ks = (slab, super-step ss, j): dims slab*128 + 16*(2*t4+ss) + 4j + {0,1},{2,3}
          const int slab = ks / 8, ss = (ks / 4) & 1, j = ks & 3;
          d0 = slab * 128 + 16 * (2 * t4 + ss) + 4 * j;
          d1 = d0 + 2;
        } else {
          d0 = ks * 16 + 2 * t4;
          d1 = d0 + 8;
        }
        qf[ksl][n][0] = qrow ? __ldg(reinterpret_cast<const uint32_t*>(qrow + d0)) : 0u;
        qf[ksl][n][1] = qrow ? __ldg(reinterpret_cast<const uint32_t*>(qrow + d1)) : 0u;
      }
    }
    if constexpr (Cfg::kQScale) {
#pragma unroll
      for (int n = 0; n < NTW; ++n) {
        if constexpr (DS == 1) {
          // the four lanes of row g hold all of its D: their fragments' maximum
          float m = 0.f;
#pragma unroll
          for (int ksl = 0; ksl < KSW; ++ksl)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const uint32_t w = qf[ksl][n][h];
              m = fmaxf(m, fmaxf(fabsf(__uint_as_float(w << 16)), fabsf(__uint_as_float(w & 0xffff0000u))));
            }
          m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
          m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
          eq[n] = q_row_exponent(m);
          sl2r[n][0] = p.sl2 * pow2f(-__shfl_sync(0xffffffffu, eq[n], 8 * t4));
          sl2r[n][1] = p.sl2 * pow2f(-__shfl_sync(0xffffffffu, eq[n], 8 * t4 + 4));
        }
        // bfloat16 pair * 2^e -> fp16 pair, exact
        const float up = pow2f(eq[n]);
#pragma unroll
        for (int ksl = 0; ksl < KSW; ++ksl)
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const uint32_t w = qf[ksl][n][h];
            qf[ksl][n][h] = pack_half2(__uint_as_float(w << 16) * up, __uint_as_float(w & 0xffff0000u) * up);
          }
      }
    }
    int lo_r[NTW][2], hi_r[NTW][2];
    float m_r[NTW][2], l_r[NTW][2];
#pragma unroll
    for (int n = 0; n < NTW; ++n) {
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const int r = (rg * NTW + n) * 8 + 2 * t4 + c;
        if (r < pc.R) {
          const int pos = pc.L - pc.qlen + r / p.G;
          hi_r[n][c] = pos;
          lo_r[n][c] = (p.window > 0) ? max(0, pos - p.window + 1) : 0;
        } else {
          hi_r[n][c] = -1;
          lo_r[n][c] = 0;
        }
        m_r[n][c] = -INFINITY;
        l_r[n][c] = 0.f;
      }
#pragma unroll
      for (int mt = 0; mt < MTW; ++mt) o[mt][n][0] = o[mt][n][1] = o[mt][n][2] = o[mt][n][3] = 0.f;
    }

    // ---- this key group's tiles of the piece: those whose ring sequence
    // number q + k is kg modulo KG. The assignment follows the ring, not the
    // piece: with a piece-local one, a piece whose length is not a multiple of
    // KG hands the following stages to the other group, and a group that
    // skips a stage's phase could pass its next wait there on a phase two
    // rounds old while that stage's load is still in flight.
    for (int k = (kg - static_cast<int>(q % KG) + KG) % KG; k < pc.ntiles; k += KG) {
      const uint32_t qq = q + k;
      const int stage = qq % NS;
      if (ok) ok = mbar_wait(full0 + 8 * stage, (qq / NS) & 1, p.timeout_ns);
      if (!ok) {
        // gave up: skip the work but keep the pair's barrier sequence, so the
        // partner warp (whose own wait may have succeeded) is never stranded
        if constexpr (DS > 1) named_bar_sync(2 + pair, DS * 32);
        continue;
      }
      const uint32_t kb = smem_u32(smem + stage * Cfg::kStageBytes);
      const uint32_t vb = kb + Cfg::kTileBytes;
      const int key0 = (pc.first_tile + k) * kTileKeys;

      // S^T = K Q^T over this warp's part of D (16 keys x 8 rows per row tile)
      float sa[NTW][4], sb[NTW][4];
#pragma unroll
      for (int n = 0; n < NTW; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e) sa[n][e] = sb[n][e] = 0.f;
      if constexpr (!FP8) {
        const int key = (lane & 7) + ((lane >> 3) & 1) * 8;
        const int srow = key * HG + th;  // 128-byte row of (key, head) in a slab
        const uint32_t rowb = kb + srow * 128;
#pragma unroll
        for (int ksl = 0; ksl < KSW; ++ksl) {
          const int ks = dh * KSW + ksl;
          const int slab = ks >> 2, chunk = (ks & 3) * 2 + (lane >> 4);
          uint32_t a[4];
          ldsm_x4(rowb + slab * Cfg::kSlabBytes + ((chunk ^ (srow & 7)) << 4), a);
#pragma unroll
          for (int n = 0; n < NTW; ++n) {
            if (ksl & 1) mma_op<BF16>(sb[n], a, qf[ksl][n][0], qf[ksl][n][1]);
            else mma_op<BF16>(sa[n], a, qf[ksl][n][0], qf[ksl][n][1]);
          }
        }
      } else {
        // rows (key g, head th) and (key g+8, head th); both have swizzle phase srow & 7
        const int srow = g * HG + th;
        const uint32_t r0 = kb + srow * 128, r8 = kb + (srow + 8 * HG) * 128;
        // super-steps of 4 k-steps: (slab, ss) = ks / 4
#pragma unroll
        for (int sup = 0; sup < KSW / 4; ++sup) {
          const int gsup = dh * (KSW / 4) + sup;
          const int slab = gsup >> 1, ss = gsup & 1;
          const int chunk = (2 * t4 + ss) ^ (srow & 7);
          uint4 w0, w8;
          asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                       : "=r"(w0.x), "=r"(w0.y), "=r"(w0.z), "=r"(w0.w)
                       : "r"(r0 + slab * Cfg::kSlabBytes + (chunk << 4)));
          asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                       : "=r"(w8.x), "=r"(w8.y), "=r"(w8.z), "=r"(w8.w)
                       : "r"(r8 + slab * Cfg::kSlabBytes + (chunk << 4)));
          const uint32_t wa[4] = {w0.x, w0.y, w0.z, w0.w};
          const uint32_t wb[4] = {w8.x, w8.y, w8.z, w8.w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int ksl = sup * 4 + j;
            uint32_t a[4];
            const uint32_t xa = byte_word_prep<Cfg::KV>(wa[j]), xb = byte_word_prep<Cfg::KV>(wb[j]);
            a[0] = byte_pair_to_half2<Cfg::KV>(xa, false);
            a[1] = byte_pair_to_half2<Cfg::KV>(xb, false);
            a[2] = byte_pair_to_half2<Cfg::KV>(xa, true);
            a[3] = byte_pair_to_half2<Cfg::KV>(xb, true);
#pragma unroll
            for (int n = 0; n < NTW; ++n) {
              if (j & 1) mma_op<BF16>(sb[n], a, qf[ksl][n][0], qf[ksl][n][1]);
              else mma_op<BF16>(sa[n], a, qf[ksl][n][0], qf[ksl][n][1]);
            }
          }
        }
      }
      float sc[NTW][4];
#pragma unroll
      for (int n = 0; n < NTW; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e) sc[n][e] = sa[n][e] + sb[n][e];
      if constexpr (DS > 1) {
        // sum the group's partial scores in part order (every warp of the group
        // evaluates the same expression, so all hold identical scores)
        // (double-buffered by the group's own tile count, so that a fast warp's
        // next tile never writes the buffer its partner is still reading)
        float* grp = xchg + (pair * 2 + ((qq / KG) & 1)) * DS * Cfg::kXchgFloats + lane * 4 * NTW;
#pragma unroll
        for (int n = 0; n < NTW; ++n)
          *reinterpret_cast<float4*>(grp + dh * Cfg::kXchgFloats + 4 * n) =
              make_float4(sc[n][0], sc[n][1], sc[n][2], sc[n][3]);
        named_bar_sync(2 + pair, DS * 32);
#pragma unroll
        for (int n = 0; n < NTW; ++n) {
          float4 t = *reinterpret_cast<const float4*>(grp + 4 * n);
#pragma unroll
          for (int part = 1; part < DS; ++part) {
            const float4 v = *reinterpret_cast<const float4*>(grp + part * Cfg::kXchgFloats + 4 * n);
            t.x += v.x; t.y += v.y; t.z += v.z; t.w += v.w;
          }
          sc[n][0] = t.x; sc[n][1] = t.y; sc[n][2] = t.z; sc[n][3] = t.w;
        }
      }
      // per row tile: mask, online softmax, P^T fragments; C layout of S^T:
      // [0]=(key g,row 2t4) [1]=(key g,row 2t4+1) [2]=(key g+8,row 2t4) [3]=(key g+8,row 2t4+1)
      uint32_t pb0[NTW], pb1[NTW];
      float al[NTW][2];
      bool rescale = false;
      // a tile every real row sees in full needs no per-key mask
      const bool interior = key0 >= pc.tile_lo_all && key0 + kTileKeys - 1 <= pc.tile_hi_all;
#pragma unroll
      for (int n = 0; n < NTW; ++n) {
        const int j0 = key0 + g, j1 = j0 + 8;
        float x[4];
        if (interior) {
          // padded rows (hi = -1) stay masked
          x[0] = hi_r[n][0] >= 0 ? sc[n][0] * sl2r[n][0] : -INFINITY;
          x[1] = hi_r[n][1] >= 0 ? sc[n][1] * sl2r[n][1] : -INFINITY;
          x[2] = hi_r[n][0] >= 0 ? sc[n][2] * sl2r[n][0] : -INFINITY;
          x[3] = hi_r[n][1] >= 0 ? sc[n][3] * sl2r[n][1] : -INFINITY;
        } else {
          x[0] = (j0 >= lo_r[n][0] && j0 <= hi_r[n][0]) ? sc[n][0] * sl2r[n][0] : -INFINITY;
          x[1] = (j0 >= lo_r[n][1] && j0 <= hi_r[n][1]) ? sc[n][1] * sl2r[n][1] : -INFINITY;
          x[2] = (j1 >= lo_r[n][0] && j1 <= hi_r[n][0]) ? sc[n][2] * sl2r[n][0] : -INFINITY;
          x[3] = (j1 >= lo_r[n][1] && j1 <= hi_r[n][1]) ? sc[n][3] * sl2r[n][1] : -INFINITY;
        }
        float mx0 = fmaxf(x[0], x[2]), mx1 = fmaxf(x[1], x[3]);
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
          mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
          mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
        }
        const float mn0 = fmaxf(m_r[n][0], mx0), mn1 = fmaxf(m_r[n][1], mx1);
        const float base0 = (mn0 == -INFINITY) ? 0.f : mn0;
        const float base1 = (mn1 == -INFINITY) ? 0.f : mn1;
        // nothing accumulated yet (m = -inf): O and l are zero, keep factor 1
        al[n][0] = (m_r[n][0] == -INFINITY) ? 1.f : ex2(m_r[n][0] - base0);
        al[n][1] = (m_r[n][1] == -INFINITY) ? 1.f : ex2(m_r[n][1] - base1);
        const float p00 = ex2(x[0] - base0), p01 = ex2(x[1] - base1);
        const float p10 = ex2(x[2] - base0), p11 = ex2(x[3] - base1);
        m_r[n][0] = mn0;
        m_r[n][1] = mn1;
        l_r[n][0] = l_r[n][0] * al[n][0] + (p00 + p10);
        l_r[n][1] = l_r[n][1] * al[n][1] + (p01 + p11);
        rescale |= (al[n][0] != 1.f || al[n][1] != 1.f);
        pb0[n] = movmatrix_trans(pack2<BF16>(p00, p01));
        pb1[n] = movmatrix_trans(pack2<BF16>(p10, p11));
      }
      if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll
        for (int mt = 0; mt < MTW; ++mt)
#pragma unroll
          for (int n = 0; n < NTW; ++n) {
            o[mt][n][0] *= al[n][0]; o[mt][n][1] *= al[n][1];
            o[mt][n][2] *= al[n][0]; o[mt][n][3] *= al[n][1];
          }
      }

      // O^T += V^T P^T over this warp's m-tiles. Keys at or past the sequence
      // end (the unwritten tail of its last block) may hold any bits, NaN
      // included: their V is zeroed so that P = 0 there never meets 0 * NaN.
      const bool tail = key0 + kTileKeys > pc.L;
      if constexpr (!FP8) {
        const int key = (lane & 7) + (lane >> 4) * 8;
        const int srow = key * HG + th;
        const uint32_t rowb = vb + srow * 128;
        // A = V^T fragment: a[0], a[1] hold keys 2t4, 2t4+1; a[2], a[3] keys 2t4+8, 2t4+9
        uint32_t vm01 = 0xffffffffu, vm23 = 0xffffffffu;
        if (tail) {
          const int k0 = key0 + 2 * t4;
          vm01 = (k0 < pc.L ? 0x0000ffffu : 0u) | (k0 + 1 < pc.L ? 0xffff0000u : 0u);
          vm23 = (k0 + 8 < pc.L ? 0x0000ffffu : 0u) | (k0 + 9 < pc.L ? 0xffff0000u : 0u);
        }
#pragma unroll
        for (int mtl = 0; mtl < MTW; ++mtl) {
          const int mt = dh * MTW + mtl;
          const int slab = mt >> 2, chunk = (mt & 3) * 2 + ((lane >> 3) & 1);
          uint32_t a[4];
          ldsm_x4_trans(rowb + slab * Cfg::kSlabBytes + ((chunk ^ (srow & 7)) << 4), a);
          if (tail) {
            a[0] &= vm01; a[1] &= vm01; a[2] &= vm23; a[3] &= vm23;
          }
#pragma unroll
          for (int n = 0; n < NTW; ++n) mma_op<BF16>(o[mtl][n], a, pb0[n], pb1[n]);
        }
      } else {
        // 32-dim group P32: lane reads 4 codes at dims 32*P32 + 4g .. +3 of keys
        // 2t4, 2t4+1, 2t4+8, 2t4+9; m-tile 2*P32 takes dims 4g (m=g) and 4g+1
        // (m=g+8), m-tile 2*P32+1 takes 4g+2 and 4g+3.
        const int kA = 2 * t4, kB = kA + 1, kC = kA + 8, kD = kA + 9;
#pragma unroll
        for (int pl = 0; pl < MTW / 2; ++pl) {
          const int P32 = dh * (MTW / 2) + pl;
          const int slab = P32 >> 2;
          const int chunk = (P32 & 3) * 2 + (g >> 2);
          const int byte = (4 * g) & 15;
          const uint32_t sb0 = vb + slab * Cfg::kSlabBytes + byte;
          uint32_t wA, wB, wC, wD;
          const int rA = kA * HG + th, rB = kB * HG + th, rC = kC * HG + th, rD = kD * HG + th;
          asm volatile("ld.shared.b32 %0, [%1];" : "=r"(wA) : "r"(sb0 + rA * 128 + ((chunk ^ (rA & 7)) << 4)));
          asm volatile("ld.shared.b32 %0, [%1];" : "=r"(wB) : "r"(sb0 + rB * 128 + ((chunk ^ (rB & 7)) << 4)));
          asm volatile("ld.shared.b32 %0, [%1];" : "=r"(wC) : "r"(sb0 + rC * 128 + ((chunk ^ (rC & 7)) << 4)));
          asm volatile("ld.shared.b32 %0, [%1];" : "=r"(wD) : "r"(sb0 + rD * 128 + ((chunk ^ (rD & 7)) << 4)));
          if (tail) {  // code 0 is the value 0 in both byte formats
            if (key0 + kA >= pc.L) wA = 0u;
            if (key0 + kB >= pc.L) wB = 0u;
            if (key0 + kC >= pc.L) wC = 0u;
            if (key0 + kD >= pc.L) wD = 0u;
          }
          wA = byte_word_prep<Cfg::KV>(wA); wB = byte_word_prep<Cfg::KV>(wB);
          wC = byte_word_prep<Cfg::KV>(wC); wD = byte_word_prep<Cfg::KV>(wD);
          const uint32_t ab01 = prmt(wA, wB, 0x5140u), ab23 = prmt(wA, wB, 0x7362u);
          const uint32_t cd01 = prmt(wC, wD, 0x5140u), cd23 = prmt(wC, wD, 0x7362u);
          uint32_t a[4];
          a[0] = byte_pair_to_half2<Cfg::KV>(ab01, false);
          a[1] = byte_pair_to_half2<Cfg::KV>(ab01, true);
          a[2] = byte_pair_to_half2<Cfg::KV>(cd01, false);
          a[3] = byte_pair_to_half2<Cfg::KV>(cd01, true);
#pragma unroll
          for (int n = 0; n < NTW; ++n) mma_op<BF16>(o[2 * pl][n], a, pb0[n], pb1[n]);
          a[0] = byte_pair_to_half2<Cfg::KV>(ab23, false);
          a[1] = byte_pair_to_half2<Cfg::KV>(ab23, true);
          a[2] = byte_pair_to_half2<Cfg::KV>(cd23, false);
          a[3] = byte_pair_to_half2<Cfg::KV>(cd23, true);
#pragma unroll
          for (int n = 0; n < NTW; ++n) mma_op<BF16>(o[2 * pl + 1][n], a, pb0[n], pb1[n]);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty0 + 8 * stage);
    }
    q += pc.ntiles;

    // ---- row sums over the lanes of each row (m is already warp-uniform per row)
#pragma unroll
    for (int n = 0; n < NTW; ++n)
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        l_r[n][0] += __shfl_xor_sync(0xffffffffu, l_r[n][0], off);
        l_r[n][1] += __shfl_xor_sync(0xffffffffu, l_r[n][1], off);
      }
    const int tid = threadIdx.x;
    const bool direct = pc.npieces == 1;
    constexpr int NT = Cfg::NT, RH = NT * 8;  // partial rows per head of a unit
    if constexpr (Cfg::kSmemMerge) {
      // ---- merge the KG key groups of each row tile through shared memory
      // (m and l are identical in the warps of a D group; warp dh = 0 posts them)
      if (g == 0 && dh == 0) {
#pragma unroll
        for (int n = 0; n < NTW; ++n) {
          float* ml = merge_ml + ((th * NT + rg * NTW + n) * KG + kg) * 16;
          ml[(2 * t4) * 2 + 0] = m_r[n][0];
          ml[(2 * t4) * 2 + 1] = l_r[n][0];
          ml[(2 * t4 + 1) * 2 + 0] = m_r[n][1];
          ml[(2 * t4 + 1) * 2 + 1] = l_r[n][1];
        }
      }
      named_bar_sync(1, Cfg::kConsumerThreads);
      {
        // this warp's weight per row: exp2(m_own - max over the key groups)
        float f_r[NTW][2];
#pragma unroll
        for (int n = 0; n < NTW; ++n)
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            const int row = 2 * t4 + c;
            float M = -INFINITY;
#pragma unroll
            for (int k = 0; k < KG; ++k)
              M = fmaxf(M, merge_ml[(((th * NT + rg * NTW + n) * KG + k) * 8 + row) * 2]);
            f_r[n][c] = (m_r[n][c] == -INFINITY) ? 0.f : ex2(m_r[n][c] - M);
          }
        // each row tile's buffer accumulates f * O one key group at a time
        const int r0 = 2 * t4, r1 = r0 + 1;
#pragma unroll 1
        for (int k = 0; k < KG; ++k) {
          if (kg == k) {
#pragma unroll
            for (int n = 0; n < NTW; ++n) {
              float* mo = merge_o + (th * NT + rg * NTW + n) * 8 * Cfg::kDP;
#pragma unroll
              for (int mtl = 0; mtl < MTW; ++mtl) {
                const int mt = dh * MTW + mtl;
                int d0, d1;  // output dims of C rows g and g+8 of m-tile mt
                if constexpr (FP8) {
                  d0 = (mt >> 1) * 32 + 4 * g + 2 * (mt & 1);
                  d1 = d0 + 1;
                } else {
                  d0 = mt * 16 + g;
                  d1 = d0 + 8;
                }
                float* a00 = mo + r0 * Cfg::kDP + d0;
                float* a10 = mo + r1 * Cfg::kDP + d0;
                float* a01 = mo + r0 * Cfg::kDP + d1;
                float* a11 = mo + r1 * Cfg::kDP + d1;
                if (k == 0) {
                  *a00 = f_r[n][0] * o[mtl][n][0]; *a10 = f_r[n][1] * o[mtl][n][1];
                  *a01 = f_r[n][0] * o[mtl][n][2]; *a11 = f_r[n][1] * o[mtl][n][3];
                } else {
                  *a00 += f_r[n][0] * o[mtl][n][0]; *a10 += f_r[n][1] * o[mtl][n][1];
                  *a01 += f_r[n][0] * o[mtl][n][2]; *a11 += f_r[n][1] * o[mtl][n][3];
                }
              }
            }
          }
          named_bar_sync(1, Cfg::kConsumerThreads);
        }
      }

      constexpr int DCH = D / 8;  // 8-dim chunks per row
      const int per_head = pc.R * DCH;
      for (int item = tid; item < HG * per_head; item += Cfg::kConsumerThreads) {
        const int hh = item / per_head, rem = item - hh * per_head;
        const int r = rem / DCH, dc = rem % DCH;
        const int rnt = hh * NT + (r >> 3), rr = r & 7;
        float M = -INFINITY;
#pragma unroll
        for (int k = 0; k < KG; ++k) M = fmaxf(M, merge_ml[((rnt * KG + k) * 8 + rr) * 2]);
        float Ls = 0.f;
#pragma unroll
        for (int k = 0; k < KG; ++k) {
          const float mk = merge_ml[((rnt * KG + k) * 8 + rr) * 2];
          if (mk != -INFINITY) Ls += ex2(mk - M) * merge_ml[((rnt * KG + k) * 8 + rr) * 2 + 1];
        }
        const float* src = merge_o + (rnt * 8 + rr) * Cfg::kDP + dc * 8;
        const float4 v0 = *reinterpret_cast<const float4*>(src);
        const float4 v1 = *reinterpret_cast<const float4*>(src + 4);
        if (direct) {
          const int i = r / p.G, hl = r % p.G;
          __half* dst = p.out + (static_cast<long long>(pc.q0 + i) * p.Hq + (pc.kh + hh) * p.G + hl) * D + dc * 8;
          const float inv = (Ls > 0.f) ? p.out_scale / Ls : 0.f;
          uint4 v;
          v.x = pack2<Cfg::QB>(v0.x * inv, v0.y * inv);
          v.y = pack2<Cfg::QB>(v0.z * inv, v0.w * inv);
          v.z = pack2<Cfg::QB>(v1.x * inv, v1.y * inv);
          v.w = pack2<Cfg::QB>(v1.z * inv, v1.w * inv);
          *reinterpret_cast<uint4*>(dst) = v;
        } else {
          const long long prow = static_cast<long long>(pc.slot) * Cfg::RP + hh * RH + r;
          float* dst = p.ws_o + prow * D + dc * 8;
          __stcg(reinterpret_cast<float4*>(dst), v0);
          __stcg(reinterpret_cast<float4*>(dst + 4), v1);
          if (dc == 0) __stcg(reinterpret_cast<float2*>(p.ws_ml + prow * 2), make_float2(M, Ls));
        }
      }
    } else {
      // ---- one key group per head: this warp's (m, l, O) are final for its
      // rows and dims, written straight from the accumulator fragments
#pragma unroll
      for (int n = 0; n < NTW; ++n)
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const int r = (rg * NTW + n) * 8 + 2 * t4 + c;
          if (r >= pc.R) continue;
          const float Ls = l_r[n][c];
          if (direct) {
            const int i = r / p.G, hl = r % p.G;
            __half* dst = p.out + (static_cast<long long>(pc.q0 + i) * p.Hq + (pc.kh + th) * p.G + hl) * D;
            const float inv = (Ls > 0.f) ? p.out_scale / Ls : 0.f;
#pragma unroll
            for (int mtl = 0; mtl < MTW; ++mtl) {
              const int mt = dh * MTW + mtl;
              if constexpr (FP8) {
                const int d0 = (mt >> 1) * 32 + 4 * g + 2 * (mt & 1);  // dims d0, d0 + 1
                *reinterpret_cast<uint32_t*>(dst + d0) =
                    pack2<Cfg::QB>(o[mtl][n][c] * inv, o[mtl][n][2 + c] * inv);
              } else {
                const int d0 = mt * 16 + g;                           // dims d0, d0 + 8
                reinterpret_cast<uint16_t*>(dst)[d0] = pack1<Cfg::QB>(o[mtl][n][c] * inv);
                reinterpret_cast<uint16_t*>(dst)[d0 + 8] = pack1<Cfg::QB>(o[mtl][n][2 + c] * inv);
              }
            }
          } else {
            const long long prow = static_cast<long long>(pc.slot) * Cfg::RP + th * RH + r;
            float* dst = p.ws_o + prow * D;
#pragma unroll
            for (int mtl = 0; mtl < MTW; ++mtl) {
              const int mt = dh * MTW + mtl;
              if constexpr (FP8) {
                const int d0 = (mt >> 1) * 32 + 4 * g + 2 * (mt & 1);
                __stcg(reinterpret_cast<float2*>(dst + d0), make_float2(o[mtl][n][c], o[mtl][n][2 + c]));
              } else {
                const int d0 = mt * 16 + g;
                __stcg(dst + d0, o[mtl][n][c]);
                __stcg(dst + d0 + 8, o[mtl][n][2 + c]);
              }
            }
            if (g == 0 && dh == 0) __stcg(reinterpret_cast<float2*>(p.ws_ml + prow * 2), make_float2(m_r[n][c], Ls));
          }
        }
    }
    if constexpr (Cfg::kSmemMerge) named_bar_sync(1, Cfg::kConsumerThreads);  // merge buffers free again
  }
  if (!ok && lane == 0) raise_error(p.error_flag, kErrTimeout);
  if (p.cluster > 1) cluster_merge_ws<D, Cfg::RP, Cfg::NT * 8, Cfg::HG, Cfg::kThreads>(p);
}

// ---------------------------------------------------------------------------
// The pieces of split unit u as the decode kernel's walk (work_next) cuts
// them: P pieces, piece 0 in slot slot0, piece k > 0 in slot slot_base + step
// * k (step 2 balanced, 1 fixed). Balanced mode restates the walk's prefix
// over the sequences (a block-wide sum of every sequence's unit_cost-charged
// span before b, and of all of them) and its chunk plan over the decode grid;
// every thread of the CTA must call it. P <= 1: nothing to merge.
template <int NW>
__device__ __forceinline__ void unit_layout(const DecodeParams& p, int u, long long (&s_red)[2][NW], int& P,
                                            long long& slot0, long long& slot_base, int& step) {
  const int b = u / p.hgn, grp = u % p.hgn;
  int L, t0, n, q0, qn;
  seq_span(p, b, false, L, t0, n, q0, qn);
  if (p.num_splits > 0) {
    const int S = p.num_splits;
    const int chunk = (n + S - 1) / S;
    P = n > 0 ? (n + chunk - 1) / chunk : 0;
    slot0 = slot_base = static_cast<long long>(u) * S;
    step = 1;
    return;
  }
  step = 2;
  long long before = 0, total = 0;
  for (int bb = threadIdx.x; bb < p.B; bb += blockDim.x) {
    int Lb, tb, nb, qb, qnb;
    seq_span(p, bb, false, Lb, tb, nb, qb, qnb);
    const long long v = nb > 0 ? static_cast<long long>(nb + p.unit_cost) * p.hgn : 0;
    total += v;
    if (bb < b) before += v;
  }
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    before += __shfl_xor_sync(0xffffffffu, before, o);
    total += __shfl_xor_sync(0xffffffffu, total, o);
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) {
    s_red[0][warp] = before;
    s_red[1][warp] = total;
  }
  __syncthreads();
  before = total = 0;
  for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) {
    before += s_red[0][w];
    total += s_red[1][w];
  }
  if (n == 0) {
    P = 0;
    slot0 = slot_base = 0;
    return;
  }
  const ChunkPlan cp = make_chunk_plan(total, p.decode_grid);
  const long long span = n + p.unit_cost;
  const long long us = before + grp * span;
  const long long rs = us + p.unit_cost, ue = us + span;
  const int cf = cp.owner(rs), cl = cp.owner(ue - 1);
  P = cl - cf + 1;
  slot_base = 2ll * cf;
  slot0 = slot_base + (cp.start(cf) < rs ? 1 : 0);
}

// The split combine's running merge of pieces k0, k0 + stride, ... (< P) of
// one item (row r of the head whose rows start at rbase, dims dim0 .. dim0 +
// 3) into (m_run, l_run, acc), in piece order; the partials of NB pieces are
// loaded at a time, all in flight at once. Piece k sits in slot slot0 (k = 0)
// or slot_base + step * k.
template <int D, int NB>
__device__ __forceinline__ void merge_pieces(const DecodeParams& p, int P, long long slot0, long long slot_base,
                                             int step, int rbase, int r, int dim0, int k0, int stride,
                                             float& m_run, float& l_run, float4& acc) {
  const int RP = p.rows_padded;
  for (; k0 < P; k0 += NB * stride) {
    float2 ml[NB];
    float4 v[NB];
#pragma unroll
    for (int j = 0; j < NB; ++j) {
      const int k = k0 + j * stride;
      if (k < P) {
        const long long sl = k == 0 ? slot0 : slot_base + static_cast<long long>(step) * k;
        ml[j] = __ldcg(reinterpret_cast<const float2*>(p.ws_ml + (sl * RP + rbase + r) * 2));
        v[j] = __ldcg(reinterpret_cast<const float4*>(p.ws_o + (sl * RP + rbase + r) * D + dim0));
      } else {
        ml[j] = make_float2(-INFINITY, 0.f);
        v[j] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
#pragma unroll
    for (int j = 0; j < NB; ++j) {
      const float mk = ml[j].x;
      if (mk == -INFINITY) continue;
      if (mk > m_run) {
        const float sc = (m_run == -INFINITY) ? 0.f : ex2(m_run - mk);
        l_run *= sc;
        acc.x *= sc; acc.y *= sc; acc.z *= sc; acc.w *= sc;
        m_run = mk;
      }
      const float w = ex2(mk - m_run);
      l_run += w * ml[j].y;
      acc.x += w * v[j].x; acc.y += w * v[j].y; acc.z += w * v[j].z; acc.w += w * v[j].w;
    }
  }
}

// ---------------------------------------------------------------------------
// Split combine: merges the fp32 (m, l, O) partials of every unit the decode
// kernel split into pieces (m in log2 units, O relative to m). Launched after
// the decode kernel with programmatic dependent launch: its CTAs may start
// while the decode grid drains and wait in griddepcontrol.wait until that grid
// has completed and its writes are visible.
//   grid (units, C, heads per tile), NT threads (256, or 512 for the
//   batch-8 kernel when a CTA holds more than 256 items): CTA (u, c, z) merges
//   head z of unit u for output dims [c*D/C, (c+1)*D/C); the host picks
//   C = D/8 (16 or more pieces per unit), D/32 (4 or more) or 1, halved
//   while the grid exceeds one CTA per SM. An item is (row, 4 dims). With more than NT items a
//   thread merges its items' pieces in order with a running max; with fewer,
//   thread t covers item t % items for pieces pg, pg+PG, ... (pg = t / items,
//   PG = NT / items) and the PG partial states are then merged in pg order.
//   Either way the result does not depend on scheduling; NB pieces' partials
//   are loaded at a time (the host takes NB = 8 when units have more than
//   four pieces, else 4, whose kernel needs fewer registers). The unit's pieces
//   and their slots are derived from the sequence lengths (inputs the decode
//   kernel does not write) before the wait, so that the first global read
//   after it is already a partial.
template <int D, int NB, int NT>
__global__ void __launch_bounds__(NT) split_combine_kernel(const DecodeParams p) {
  __shared__ float s_m[NT], s_l[NT];
  __shared__ float4 s_o[NT];
  __shared__ long long s_red[2][NT / 32];
  // the next launch in the stream may be scheduled now (it waits for this
  // grid in its own griddepcontrol.wait before touching global memory): its
  // CTAs take the SMs the decode grid leaves while this grid, resident beside
  // it, merges (measured on GB300, D=256 GQA 6:1: B = 1 / 8 / 32 11.95 /
  // 28.13 / 82.42 -> 11.65 / 27.82 / 82.16 us per call in a loop of calls;
  // e4m3 B = 32 52.0 -> 52.4)
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int u = blockIdx.x;
  int P, step;
  long long slot0, slot_base;
  unit_layout(p, u, s_red, P, slot0, slot_base, step);
  const int b = u / p.hgn;
  int q0, qn;
  seq_queries(p, b, false, q0, qn);
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (P <= 1) return;
  const int R = p.R;
  // blockIdx.z: head of the unit's head group; its rows start at z * rows_head
  const int kh = (u % p.hgn) * p.hg + blockIdx.z;
  const int rbase = blockIdx.z * p.rows_head;
  const int live_rows = p.G * qn;  // rows of the sequence's query tokens
  // blockIdx.y: which D / gridDim.y output dims; an item is (row, 4 dims)
  const int dims_cta = D / gridDim.y, slices = dims_cta / 4;
  const int items = R * slices;
  const int t = threadIdx.x;
  auto store = [&](int r, int dim0, float L, float4 o) {
    const float inv = (L > 0.f) ? p.out_scale / L : 0.f;
    const int i = r / p.G, hl = r % p.G;
    __half* dst = p.out + (static_cast<long long>(q0 + i) * p.Hq + kh * p.G + hl) * D + dim0;
    uint2 o2;
    if (p.out_bf16) {
      o2.x = pack_bf162(o.x * inv, o.y * inv);
      o2.y = pack_bf162(o.z * inv, o.w * inv);
    } else {
      o2.x = pack_half2(o.x * inv, o.y * inv);
      o2.y = pack_half2(o.z * inv, o.w * inv);
    }
    *reinterpret_cast<uint2*>(dst) = o2;
  };

  if (items > NT) {
    // many items, few pieces each: one thread per item, all pieces in order
    for (int item = t; item < items; item += NT) {
      const int r = item / slices, dim0 = blockIdx.y * dims_cta + (item % slices) * 4;
      if (r >= live_rows) continue;
      float m_run = -INFINITY, l_run = 0.f;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      merge_pieces<D, NB>(p, P, slot0, slot_base, step, rbase, r, dim0, 0, 1, m_run, l_run, acc);
      store(r, dim0, l_run, acc);
    }
    return;
  }
  // few items, possibly many pieces: PG thread groups take interleaved
  // pieces, then the groups merge in group order (deterministic)
  const int PG = NT / items;
  const int item = t % items, pg = t / items;
  const int r = item / slices, dim0 = blockIdx.y * dims_cta + (item % slices) * 4;
  const bool live = r < live_rows;
  float m_run = -INFINITY, l_run = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  if (pg < PG && live)
    merge_pieces<D, NB>(p, P, slot0, slot_base, step, rbase, r, dim0, pg, PG, m_run, l_run, acc);
  s_m[t] = m_run;
  s_l[t] = l_run;
  s_o[t] = acc;
  __syncthreads();
  if (pg != 0 || t >= items || !live) return;
  float M = -INFINITY;
  for (int g2 = 0; g2 < PG; ++g2) M = fmaxf(M, s_m[g2 * items + item]);
  float L = 0.f;
  float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int g2 = 0; g2 < PG; ++g2) {
    const float mg = s_m[g2 * items + item];
    if (mg == -INFINITY) continue;
    const float w = ex2(mg - M);
    L += w * s_l[g2 * items + item];
    const float4 a = s_o[g2 * items + item];
    o.x += w * a.x; o.y += w * a.y; o.z += w * a.z; o.w += w * a.w;
  }
  store(r, dim0, L, o);
}

}  // namespace pd
