// decode_tci8.cuh -- paged decode attention for int8 caches on the
// 5th-generation tensor cores (tcgen05, accumulators in tensor memory), for
// units with 9 to 32 query rows per KV head (speculative verify, wide GQA).
//
// Same method, work split, rings, producers and merges as the e4m3 kernel of
// decode_tc8.cuh (the per-head paged decode of opengfx1030/vllm-rdna pull
// request #33, "Purpose"); the products run on fp16 operands
// (tcgen05.mma kind::f16, fp32 accumulation):
//  * The softmax warps widen the int8 codes to fp16 exactly. K of a block
//    goes into tensor memory as the A operand of S^T (lane = key, the packed
//    fp16 pairs of its row in D / 2 columns, two buffers), one block ahead of
//    its scores, each code x as the integer x + 1152 (widen_i8x16_offset): the
//    offset adds 1152 * sum(q) to every score of a row, a constant per row
//    that the score step subtracts again (kRowCf) and to which the softmax is
//    blind in any case. V of a block goes into an fp16 shared-memory buffer
//    laid out as the MN-major A operand of O^T += V^T P^T (128-byte swizzle,
//    64-dim slabs), each code as x itself (widen_i8x16). An int8 ring stage
//    is released as soon as it is widened.
//  * q is one fp16 term, scaled per row by a power of two so that its largest
//    |q| lies in [2^14, 2^15) (exact for an fp16 q; a bfloat16 q keeps its 8
//    significant bits), the factor folded into the row's score factor.
//  * The weights P are one fp16 term (at most 2^8) and the row sums add the
//    rounded weights, so each output row is a convex combination of the V rows
//    under exactly the weights the product used.
//  * S^T [128 keys x 32 rows] = K Q^T; O^T [D x 32 rows] accumulates in tensor
//    memory, output dims 128 h .. 128 h + 127 in columns kColO + 32 h.
//  * Every wait is bounded; after a timeout each role stops waiting and
//    issuing but keeps the softmax warps' named-barrier sequence, so the CTA
//    always reaches its exit, where the tensor memory is freed.
#pragma once
#include "decode_tc8.cuh"

namespace pd {

template <int D_, bool QB_ = false, int NG_ = 4>
struct Tci8 {
  static constexpr int D = D_;
  static constexpr bool QB = QB_;                   // q and out in bfloat16 (else fp16)
  static constexpr int NG = NG_;                    // softmax groups = 8-row tiles of a unit (1 to 4)
  static constexpr int kSlabs = D / 128;            // 128-byte slabs of an int8 key row; 128-dim halves of O^T
  static constexpr int kBlkTiles = 8;               // 16-key tiles per 128-key block
  static constexpr int kSlabBlk = 128 * 128;        // one slab of a block: [128 keys][128 B]
  static constexpr int kKBlk = kSlabs * kSlabBlk;   // int8 K (or V) of one block
  static constexpr int NBK = D == 256 ? 2 : 4;      // int8 K ring stages
  static constexpr int NBV = D == 256 ? 2 : 4;      // int8 V ring stages
  static constexpr int kTileBox = 16 * 128;         // one TMA box: 16 keys x 128 bytes
  static constexpr int kN = 32;                     // query rows per unit on the N side
  static constexpr int kChunks = D / 16;            // 16-code chunks of a key row
  static constexpr int kV16Slab = 128 * 128;        // fp16 V, 64 dims of a block: [128 keys][128 B]
  static constexpr int kV16Bytes = (D / 64) * kV16Slab;
  static constexpr int kQSlab = kN * 128;           // fp16 q, 64 dims: [32 rows][128 B]
  static constexpr int kQBytes = (D / 64) * kQSlab;
  static constexpr int kPtBytes = 128 * kN * 2;     // fp16 P^T: [128 keys][32 rows], MN-major
  static constexpr int kGroupRows = 8;              // query rows per softmax group
  static constexpr int kSoftThreads = 128 * NG;     // softmax warps 0 .. 4 NG - 1
  static constexpr int kThreads = kSoftThreads + 96;  // then the K and V producers and the MMA warp
  static constexpr int kProducerWarp = 4 * NG, kMmaWarp = 4 * NG + 2;
  static constexpr int kBarAll = NG + 1;            // named barrier of every softmax thread (1..NG: groups)
  static constexpr int kColS = 0;                   // S^T, two buffers of kN columns
  static constexpr int kColO = 2 * kN;              // O^T, kSlabs x kN columns
  static constexpr int kColK = kColO + kSlabs * kN;   // fp16 K (A of S^T), two buffers of D / 2 columns
  static constexpr int kTmemCols = D == 256 ? 512 : 256;
  static constexpr uint32_t kIdescS = idesc_f16(128, kN, false, false);  // A (tensor memory), B (q) K-major
  static constexpr uint32_t kIdescO = idesc_f16(128, kN, true, true);    // A (V^T), B (P^T) MN-major
  static constexpr float kRaise = 4.f;              // running max raised past this gap (log2)
  static constexpr int kUnitCost = 24;              // a piece's fixed cost in 16-key tiles (balanced split)
  static constexpr float kBias = 4.f;               // weights are 2^(x - m + kBias) <= 2^8
  static constexpr int kBarKReady = kBarSEmpty;     // the K buffers in tensor memory (two barriers)

  static constexpr int kOffV = NBK * kKBlk;
  static constexpr int kOffV16 = kOffV + NBV * kKBlk;
  static constexpr int kOffQ = kOffV16 + kV16Bytes;
  static constexpr int kOffPt = kOffQ + kQBytes;
  static constexpr int kOffRed = kOffPt + kPtBytes;        // float [NG groups][4 warps][8 rows]
  static constexpr int kRowWords = 8 * 32;                 // row state: 8 arrays of 32 words
  static constexpr int kOffRow = kOffRed + NG * 4 * kGroupRows * 4;
  // Cluster merge: each CTA stages its partial (m, l) here and its partial O
  // rows [32][D] fp32 at offset 0, over the K ring, idle once the piece is done.
  static constexpr int kOffStageMl = kOffRow + kRowWords * 4;  // float2 [32 rows]
  static constexpr int kOffBars = kOffStageMl + 32 * 8;
  static constexpr int kBars = 2 * NBK + 2 * NBV + 8;
  static constexpr int kOffTmem = kOffBars + kBars * 8;
  static constexpr int kOffPre = kOffTmem + 16;
  static constexpr int kSmemBytes = kOffPre + (kMaxAutoB + 1) * 4 + 1024;  // + alignment slack
  static_assert(D == 128 || D == 256, "head size 128 or 256");
  static_assert(NG >= 1 && NG <= 4, "one to four 8-row tiles per unit");
  static_assert(kOffV % 1024 == 0 && kOffV16 % 1024 == 0 && kOffQ % 1024 == 0 && kOffPt % 1024 == 0,
                "tensor-core operands start on 1024-byte swizzle atoms");
  static_assert(kOffRow % 16 == 0, "row state read as float4");
  static_assert(kColK + 2 * (D / 2) <= kTmemCols, "tensor-memory columns");
  static_assert(kSmemBytes <= 227 * 1024, "one CTA per SM");
  static_assert(kN * D * 4 <= NBK * kKBlk, "the staged O rows fit over the K ring");
};

__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr)
               : "memory");
  return v;
}
__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

// Sixteen int8 codes (four words, lowest byte first) to sixteen fp16 values,
// exactly (h[k] holds codes 2k and 2k + 1, the lower one in the low half).
// The code x, offset to x + 128 in [0, 255] by flipping its sign bit, becomes
// the low byte of an fp16 whose high byte is 0x64: that is 1024 + x + 128 =
// x + 1152, an integer below 2048 and so exact (widen_i8x16_offset stops
// here); subtracting 1152 leaves the integer x, exactly (fp16 represents every
// integer of magnitude at most 2048).
__device__ __forceinline__ void widen_i8x16_offset(const uint4& w, uint32_t (&h)[8]) {
  const uint32_t in[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const uint32_t u = in[k] ^ 0x80808080u;
    h[2 * k] = prmt(u, 0x64646464u, 0x4140u);
    h[2 * k + 1] = prmt(u, 0x64646464u, 0x4342u);
  }
}
__device__ __forceinline__ void widen_i8x16(const uint4& w, uint32_t (&h)[8]) {
  const uint32_t in[4] = {w.x, w.y, w.z, w.w};
  const uint32_t off2 = 0x64806480u;  // 1152 in both fp16 halves
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const uint32_t u = in[k] ^ 0x80808080u;
    const uint32_t lo = prmt(u, 0x64646464u, 0x4140u), hi = prmt(u, 0x64646464u, 0x4342u);
    const __half2 a = __hsub2(*reinterpret_cast<const __half2*>(&lo), *reinterpret_cast<const __half2*>(&off2));
    const __half2 b = __hsub2(*reinterpret_cast<const __half2*>(&hi), *reinterpret_cast<const __half2*>(&off2));
    h[2 * k] = *reinterpret_cast<const uint32_t*>(&a);
    h[2 * k + 1] = *reinterpret_cast<const uint32_t*>(&b);
  }
}

// The softmax warps (NG groups of four; thread i of a group owns TMEM lane i:
// key i of a block for S^T and K, output dims i and i + 128 for O^T; group g
// owns query rows 8 g .. 8 g + 7). Besides the softmax they widen the int8
// operands: K chunk c (16 codes) of a key row is widened by group c % NG, V
// chunk c by group (kChunks + c) % NG, which evens out each group's share of
// the 2 kChunks chunks of a key.
template <class T>
__device__ __forceinline__ void softmax_role_i8(const DecodeParams& p, const int* s_pre, WorkIter& it, Piece& pc,
                                                uint8_t* smem, uint32_t sbase, uint32_t tmem, bool& ok) {
  constexpr int D = T::D, NBK = T::NBK, NBV = T::NBV, S = T::kSlabs, NR = T::kGroupRows, NG = T::NG;
  constexpr int NST = T::kSoftThreads, NCH = T::kChunks, PER = (NCH + NG - 1) / NG;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = warp >> 2;              // row group
  const int key = tid & 127;            // TMEM lane of this thread
  const int rb = NR * g;                // first row of this group
  const int swz = key & 7;              // 128-byte swizzle of this key's rows
  const int v_first = ((g - NCH) % NG + NG) % NG;  // first V chunk of this group
  float* rf = reinterpret_cast<float*>(smem + T::kOffRow);
  int* ri = reinterpret_cast<int*>(smem + T::kOffRow);
  float* red = reinterpret_cast<float*>(smem + T::kOffRed) + 4 * NR * g;  // [4 warps][8 rows]
  const uint32_t fullk0 = sbase + T::kOffBars, emptyk0 = fullk0 + 8 * NBK;
  const uint32_t fullv0 = emptyk0 + 8 * NBK, emptyv0 = fullv0 + 8 * NBV, bx = emptyv0 + 8 * NBV;
  auto bar = [&](int i) -> uint32_t { return bx + 8 * i; };
  const uint32_t tl = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);  // this warp's TMEM lanes
  const uint32_t qs = sbase + T::kOffQ, pt = sbase + T::kOffPt, v16 = sbase + T::kOffV16;
  uint32_t bq = 0;

  // K of block b (ring stage b % NBK): this key's chunks c = g, g + NG, ...
  // widened (offset by 1152) into the block's tensor-memory buffer (b & 1),
  // columns 8 c .. 8 c + 7; then the ring stage is released and the buffer
  // marked ready. The buffer last held block b - 2, whose S^T this warp has
  // already waited for.
  auto widen_k = [&](uint32_t b) {
    const int st = b % NBK;
    if (ok) ok = mbar_wait(fullk0 + 8 * st, (b / NBK) & 1, p.timeout_ns);
    ok = __all_sync(0xffffffffu, ok);  // tcgen05.st is warp-collective
    if (ok) {
      const uint32_t src = sbase + st * T::kKBlk + key * 128;
      const uint32_t dst = tl + T::kColK + (b & 1) * (D / 2);
#pragma unroll
      for (int k = 0; k < PER; ++k) {
        const int c = g + NG * k;
        if (c < NCH) {  // warp-uniform
          uint32_t h[8];
          widen_i8x16_offset(ld_shared_v4(src + (c >> 3) * T::kSlabBlk + (((c & 7) ^ swz) << 4)), h);
          tmem_st8u(dst + 8 * c, h);
        }
      }
      tmem_wait_st();
    }
    tc_fence_before();
    __syncwarp();
    if (ok && lane == 0) {
      mbar_arrive(emptyk0 + 8 * st);
      mbar_arrive(bar(T::kBarKReady + (b & 1)));
    }
  };
  // V of block b (ring stage b % NBV): this key's chunks c = v_first, + NG, ...
  // widened into the fp16 V buffer (slab c / 4 of 64 dims, the key's 128-byte
  // row, 16-byte chunks 2 (c % 4) and 2 (c % 4) + 1 in the 128-byte swizzle);
  // then the ring stage is released. The P.V product of block b - 1, the last
  // reader of the buffer, has completed.
  auto widen_v = [&](uint32_t b) {
    const int st = b % NBV;
    if (ok) ok = mbar_wait(fullv0 + 8 * st, (b / NBV) & 1, p.timeout_ns);
    if (ok) {
      const uint32_t src = sbase + T::kOffV + st * T::kKBlk + key * 128;
#pragma unroll
      for (int k = 0; k < PER; ++k) {
        const int c = v_first + NG * k;
        if (c < NCH) {
          uint32_t h[8];
          widen_i8x16(ld_shared_v4(src + (c >> 3) * T::kSlabBlk + (((c & 7) ^ swz) << 4)), h);
          const uint32_t row = v16 + (c >> 2) * T::kV16Slab + key * 128;
          st_shared_v4(row + (((2 * (c & 3)) ^ swz) << 4), h[0], h[1], h[2], h[3]);
          st_shared_v4(row + (((2 * (c & 3) + 1) ^ swz) << 4), h[4], h[5], h[6], h[7]);
        }
      }
    }
    __syncwarp();
    if (ok && lane == 0) mbar_arrive(emptyv0 + 8 * st);
  };
  // A piece's q (the B operand of S^T: fp16, K-major, 128-byte swizzle, 64-dim
  // slabs of [32 rows][128 B]), row score factors and visible key limits; the
  // previous piece's S^T products are complete (its softmax read them all).
  // Item t < 256: row t / 8, dims [(t % 8) D / 8, (t % 8 + 1) D / 8).
  auto q_setup = [&](const Piece& pq) {
    for (int item = tid; item < 256; item += NST) {
      const int r = item >> 3, part = item & 7;
      constexpr int NW = D / 64;  // 8-dim pieces per item
      const __half* qrow = nullptr;
      if (r < pq.R) {
        const int i = r / p.G, hl = r % p.G;
        qrow = p.q + (static_cast<long long>(pq.q0 + i) * p.Hq + pq.kh * p.G + hl) * D;
      }
      uint4 qv[NW];
      float mx = 0.f;
#pragma unroll
      for (int c = 0; c < NW; ++c) {
        qv[c] = qrow ? __ldg(reinterpret_cast<const uint4*>(qrow + part * (D / 8) + 8 * c))
                     : make_uint4(0u, 0u, 0u, 0u);
        const uint32_t w[4] = {qv[c].x, qv[c].y, qv[c].z, qv[c].w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float2 f = pair_to_float2<T::QB>(w[k]);
          mx = fmaxf(mx, fmaxf(fabsf(f.x), fabsf(f.y)));
        }
      }
#pragma unroll
      for (int o = 1; o < 8; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      // 2^e with the row's largest |q| * 2^e in [2^14, 2^15), e held to
      // [-126, 126] so that 2^e and 2^-e stay normal floats
      const int e = mx > 0.f ? max(-126, min(126, 141 - static_cast<int>((__float_as_uint(mx) >> 23) & 255u)))
                             : 0;
      const float up = __uint_as_float(static_cast<uint32_t>(127 + e) << 23);
      float qsum = 0.f;  // the row's sum of its fp16 q values (for the K offset)
#pragma unroll
      for (int c = 0; c < NW; ++c) {
        const int d0 = part * (D / 8) + 8 * c;
        const uint32_t w[4] = {qv[c].x, qv[c].y, qv[c].z, qv[c].w};
        uint32_t h[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float2 f = pair_to_float2<T::QB>(w[k]);
          h[k] = pack_half2(f.x * up, f.y * up);
          const float2 hq = __half22float2(*reinterpret_cast<const __half2*>(&h[k]));
          qsum += hq.x + hq.y;
        }
        st_shared_v4(qs + (d0 >> 6) * T::kQSlab + r * 128 + ((((d0 & 63) >> 3) ^ (r & 7)) << 4), h[0], h[1], h[2],
                     h[3]);
      }
#pragma unroll
      for (int o = 1; o < 8; o <<= 1) qsum += __shfl_xor_sync(0xffffffffu, qsum, o);
      if (part == 0) {
        int lo = 0, hi = -1;
        if (r < pq.R) {
          hi = pq.L - pq.qlen + r / p.G;
          lo = p.window > 0 ? max(0, hi - p.window + 1) : 0;
        }
        const float fsl = r < pq.R ? p.sl2 * __uint_as_float(static_cast<uint32_t>(127 - e) << 23) : 0.f;
        rf[kRowFsl * 32 + r] = fsl;
        rf[kRowCf * 32 + r] = -1152.f * qsum * fsl;  // minus the K offset's share of every score
        rf[kRowMu * 32 + r] = -INFINITY;
        ri[kRowLo * 32 + r] = lo;
        ri[kRowHi * 32 + r] = hi;
      }
    }
    fence_proxy_async_smem();
  };

  while (tc_next_piece<T>(p, s_pre, it, pc)) {
    const int nblk = (pc.ntiles + T::kBlkTiles - 1) / T::kBlkTiles;
    q_setup(pc);
    named_bar_sync(T::kBarAll, NST);
    if (tid == 0) mbar_arrive(bar(kBarQFull));
    float fs[NR];  // score factor of each row of this group
#pragma unroll
    for (int r = 0; r < NR; ++r) fs[r] = rf[kRowFsl * 32 + rb + r];
    float lp[NR];  // this key lane's share of each row's weight sum
#pragma unroll
    for (int r = 0; r < NR; ++r) lp[r] = 0.f;
    widen_k(bq);

    for (int i = 0; i < nblk; ++i) {
      const uint32_t b = bq + i;
      const int sb = b & 1;
      const int key0 = (pc.first_tile + T::kBlkTiles * i) * kTileKeys;
      const int nvalid = min(128, kTileKeys * (pc.ntiles - T::kBlkTiles * i));  // keys loaded
      // ---- the next block's K goes into the other buffer while S^T of this
      // one is computed
      if (i + 1 < nblk) widen_k(b + 1);
      // ---- this key's scores for the group's 8 rows
      float x[NR];
      if (ok) ok = mbar_wait(bar(kBarSFull + sb), (b >> 1) & 1, p.timeout_ns);
      ok = __all_sync(0xffffffffu, ok);  // tcgen05.ld is warp-collective
      tc_fence_after();
      if (ok) {
        tmem_ld8(tl + T::kColS + T::kN * sb + rb, x);
        tmem_wait_ld();
      } else {
#pragma unroll
        for (int r = 0; r < NR; ++r) x[r] = 0.f;
      }
      float cf[NR];  // score offset of each row (re-read: registers are scarce)
#pragma unroll
      for (int k = 0; k < NR / 4; ++k) {
        const float4 f = reinterpret_cast<const float4*>(rf + kRowCf * 32 + rb)[k];
        cf[4 * k] = f.x; cf[4 * k + 1] = f.y; cf[4 * k + 2] = f.z; cf[4 * k + 3] = f.w;
      }
      tc_scale_mask<T, true>(x, fs, cf, key0, nvalid, pc, ri, rb, key);
      float mu[NR];
      const bool rescale = tc_raise_max<T>(x, mu, rf, ri, red, g, warp, lane);
      // ---- weights 2^(x - mu + kBias) (<= 2^8) rounded to fp16, and the row
      // sums of the rounded weights
      uint32_t pw[NR / 2];
#pragma unroll
      for (int k = 0; k < NR / 2; ++k) {
        const float a = ex2(x[2 * k] - (mu[2 * k] == -INFINITY ? 0.f : mu[2 * k] - T::kBias));
        const float c = ex2(x[2 * k + 1] - (mu[2 * k + 1] == -INFINITY ? 0.f : mu[2 * k + 1] - T::kBias));
        pw[k] = pack_half2(a, c);
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&pw[k]));
        x[2 * k] = f.x;
        x[2 * k + 1] = f.y;
      }
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
#pragma unroll
        for (int h = 0; h < S; ++h) {
          float o[NR];
          tmem_ld8(tl + T::kColO + T::kN * h + rb, o);
          tmem_wait_ld();
#pragma unroll
          for (int r = 0; r < NR; ++r) o[r] *= rf[kRowAl * 32 + rb + r];
          tmem_st8(tl + T::kColO + T::kN * h + rb, o);
        }
        tmem_wait_st();
      }
      // ---- P^T: this key's 8 row weights are the 16-byte chunk g of its
      // 64-byte row (k = key) of an MN-major operand in the 64-byte swizzle
      // layout (8-key atoms of 512 bytes, chunk ^= (key >> 1) & 3)
      st_shared_v4(pt + (key >> 3) * 512 + (key & 7) * 64 + ((g ^ ((key >> 1) & 3)) << 4), pw[0], pw[1], pw[2],
                   pw[3]);
      widen_v(b);
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (ok && lane == 0) mbar_arrive(bar(kBarPFull));
    }
    bq += nblk;

    // ---- epilogue: O^T (this thread: dims key, key + 128) of the group's rows
    if (ok) ok = mbar_wait(bar(kBarPvDone), (bq - 1) & 1, p.timeout_ns);
    ok = __all_sync(0xffffffffu, ok);
    tc_fence_after();
    float o[S][NR];
#pragma unroll
    for (int h = 0; h < S; ++h) {
      if (ok) {
        tmem_ld8(tl + T::kColO + T::kN * h + rb, o[h]);
        tmem_wait_ld();
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

template <class T>
__global__ void __launch_bounds__(T::kThreads, 1)
    decode_tci8_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                       const DecodeParams p) {
  constexpr int D = T::D, NBK = T::NBK, NBV = T::NBV;
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
      mbar_init(emptyk0 + 8 * s, 4 * T::NG);  // the widening softmax warps
    }
    for (int s = 0; s < NBV; ++s) {
      mbar_init(fullv0 + 8 * s, 1);
      mbar_init(emptyv0 + 8 * s, 4 * T::NG);
    }
    mbar_init(bar(kBarSFull), 1);
    mbar_init(bar(kBarSFull + 1), 1);
    mbar_init(bar(T::kBarKReady), 4 * T::NG);
    mbar_init(bar(T::kBarKReady + 1), 4 * T::NG);
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
  for (int i = threadIdx.x; i < T::kPtBytes / 16; i += T::kThreads)
    st_shared_v4(sbase + T::kOffPt + 16 * i, 0u, 0u, 0u, 0u);
  fence_proxy_async_smem();
  // a CTA of a cluster that gets no piece contributes nothing to the merge
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
      const uint32_t qb = sbase + T::kOffQ, pt = sbase + T::kOffPt, v16 = sbase + T::kOffV16;
      while (work_next(p, s_pre, it, pc)) {
        if (pc.ntiles == 0) continue;
        const int nblk = (pc.ntiles + T::kBlkTiles - 1) / T::kBlkTiles;
        if (ok) ok = mbar_wait(bar(kBarQFull), pq & 1, p.timeout_ns);
        ++pq;
        tc_fence_after();
        for (int i = 0; i <= nblk; ++i) {
          if (i < nblk) {  // S^T of block i = K Q^T, K from its tensor-memory buffer
            const uint32_t b = bq + i;
            const int sb = b & 1;
            if (ok) ok = mbar_wait(bar(T::kBarKReady + sb), (b >> 1) & 1, p.timeout_ns);
            tc_fence_after();
            if (ok) {
#pragma unroll
              for (int ks = 0; ks < D / 16; ++ks)
                mma_f16_ts(tmem + T::kColS + T::kN * sb, tmem + T::kColK + sb * (D / 2) + 8 * ks,
                           sdesc_sw128(qb + (ks >> 2) * T::kQSlab + (ks & 3) * 32), T::kIdescS, ks != 0 ? 1u : 0u);
              mma_commit(bar(kBarSFull + sb));
              any = true;
            }
          }
          if (i >= 1) {  // O^T += V^T P^T of block i - 1 (fp16 V, MN-major)
            const uint32_t b = bq + i - 1;
            if (ok) ok = mbar_wait(bar(kBarPFull), b & 1, p.timeout_ns);
            tc_fence_after();
            if (ok) {
#pragma unroll
              for (int h = 0; h < T::kSlabs; ++h)
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                  mma_f16_ss(tmem + T::kColO + T::kN * h,
                             sdesc_sw128_mn16(v16 + 2 * h * T::kV16Slab + kk * 2048, T::kV16Slab),
                             sdesc_sw64_mn16(pt + kk * 1024), T::kIdescO, (i > 1 || kk > 0) ? 1u : 0u);
              mma_commit(bar(kBarPvDone));
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
    softmax_role_i8<T>(p, s_pre, it, pc, smem, sbase, tmem, ok);
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

// Host launch of the int8 tensor-core decode (one CTA per SM), with
// programmatic dependent launch and, for a cluster-merged fixed split,
// clusters of p.cluster CTAs; sets the shared-memory opt-in once per context.
template <class T>
cudaError_t launch_tci8(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeParams& p, int grid,
                        cudaStream_t stream) {
  static unsigned long long attr_ctx[64] = {};
  const cudaError_t e = once_per_context(attr_ctx, [] {
    return set_kernel_attributes(decode_tci8_kernel<T>, T::kSmemBytes);
  });
  if (e != cudaSuccess) return e;
  return launch_pdl(decode_tci8_kernel<T>, grid, T::kThreads, T::kSmemBytes, stream, p.cluster, tk, tv, p);
}

template <class T>
bool shape_tci8(int nt, KernelShape* out) {
  out->threads = T::kThreads;
  out->smem_bytes = T::kSmemBytes;
  out->rows_padded = 8 * nt;
  out->ctas_per_sm = 1;
  out->heads = 1;
  out->unit_cost = T::kUnitCost;
  out->fixed_pieces = 1;
  static unsigned long long ctx_done[64] = {};
  static int cache[64][kMaxCluster + 1] = {};
  max_active_clusters(decode_tci8_kernel<T>, T::kThreads, T::kSmemBytes, ctx_done, cache, out->max_clusters);
  return true;
}

}  // namespace pd
