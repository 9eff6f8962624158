/*
 * pdecode.h -- C ABI of libpdecode: paged split-K decode attention on one
 * NVIDIA GB300 (sm_103a).
 *
 * What the library computes follows opengfx1030/vllm-rdna pull request #33
 * ("Paged split-K decode"):
 *   - "Purpose": a per-head decode over a paged KV cache -- page lookups
 *     through a block table, scores scale * q . k, online softmax, P.V, and
 *     split-K partials merged by a combine; fp16, fp8 and int8 KV share the body;
 *     every launch runs on the caller's current stream;
 *   - "What changed vs the old #33 diff": an empty key range never enters the
 *     P.V loop (empty rows are zero);
 *   - "Test Plan" step 2: the decode cells -- writer layout, empty rows are
 *     zero, a custom scale written into a caller-owned `out`, a paged sliding
 *     window, multi-token (speculative verify) queries, split decode;
 *   - "Test Result": the split-K schedule must agree with a one-shot fp64
 *     reference.
 *
 * Readings where the page is silent:
 *   - seq_lens[b] counts every cached key of sequence b, including its qlen
 *     query tokens; query token i sits at position p = seq_lens[b] - qlen + i
 *     and sees keys j <= p (causal among the query tokens);
 *   - window W > 0 keeps keys p - W + 1 <= j <= p; W <= 0 disables it;
 *   - query head h reads KV head h / (Hq / Hkv);
 *   - a row with no visible key is written as zeros.
 *
 * Conventions shared by every entry point:
 *   - All tensor pointers are DEVICE pointers owned by the caller, contiguous
 *     and row-major, on the device that is current when the call is made. The
 *     library never allocates, frees or synchronises; it launches on `stream`
 *     (a cudaStream_t; NULL = the legacy default stream) and returns at once.
 *   - Host-checkable problems are reported through the return value before
 *     anything is launched. PD_ERR_CUDA means a launch or runtime call failed;
 *     the library only peeks at the runtime's last error, so the caller's
 *     cudaGetLastError() still returns the CUDA error.
 *   - Data errors that only the device can see (a block id outside
 *     [0, num_blocks), a seq_len outside [0, max_blocks_per_seq*block_size],
 *     a pipeline wait that ran past its time limit) never trap: the kernel
 *     sets a bit of *error_flag (if error_flag is not NULL) with atomicOr and
 *     carries on; the affected rows are then unspecified. The caller clears
 *     the flag.
 *   - There is no CPU fallback and no alternative back end: shapes the
 *     kernels do not implement return PD_ERR_UNSUPPORTED.
 */
#ifndef PDECODE_H
#define PDECODE_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define PD_API __attribute__((visibility("default")))
#else
#define PD_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  PD_OK = 0,
  PD_ERR_NULL = 1,        /* a required pointer is NULL */
  PD_ERR_SHAPE = 2,       /* sizes are inconsistent or out of range */
  PD_ERR_DTYPE = 3,       /* unknown KV dtype */
  PD_ERR_UNSUPPORTED = 4, /* legal, but no kernel here implements it */
  PD_ERR_ALIGN = 5,       /* a pointer is not 16-byte aligned */
  PD_ERR_WORKSPACE = 6,   /* workspace missing or smaller than pd_workspace_bytes */
  PD_ERR_CUDA = 7         /* a CUDA runtime call or launch failed */
} pd_status;

typedef enum {
  PD_KV_F16 = 0,       /* K and V caches hold IEEE binary16 */
  PD_KV_FP8_E4M3 = 1,  /* K and V caches hold OCP e4m3fn codes; value = decode(code) * scale */
  PD_KV_INT8 = 2,      /* K and V caches hold int8 two's-complement codes; value = code * scale */
  PD_KV_BF16 = 3,      /* K and V caches, q and out hold bfloat16 (scales ignored); the products
                          run on bfloat16 tensor-core operands (P rounded to bfloat16) */
  PD_KV_FP8_E4M3_BF16 = 4, /* e4m3fn caches as PD_KV_FP8_E4M3, q and out (and the writer's new
                              tokens) in bfloat16: each q row is scaled by a power of two into
                              fp16 exactly and the products run as for an fp16 q */
  PD_KV_INT8_BF16 = 5  /* int8 caches as PD_KV_INT8, q and out (and new tokens) in bfloat16 */
} pd_kv_dtype;

/* Bits written into *error_flag by the device. */
#define PD_DEVERR_BLOCK_ID 1u /* a block_table entry used by the call is outside [0, num_blocks) */
#define PD_DEVERR_SEQ_LEN 2u  /* a seq_len is negative or above max_blocks_per_seq*block_size */
#define PD_DEVERR_TIMEOUT 4u  /* a pipeline wait ran past its limit; the call gave up */
#define PD_DEVERR_SLOT 8u     /* write_kv_cache: a slot at or beyond num_blocks*block_size */
#define PD_DEVERR_QUERY_START 16u /* decode_paged_varlen: a sequence's query range is malformed */

/* Shapes of one call.
 *   B                  number of sequences (rows of block_table / seq_lens)
 *   Hq, Hkv            query and KV heads; Hq % Hkv == 0
 *   D                  head size; the kernels implement 128 and 256
 *   block_size         keys per cache block; a multiple of 16
 *   num_blocks         blocks in each of the K and V caches
 *   max_blocks_per_seq columns of block_table
 *   kv_dtype           pd_kv_dtype
 *   k_scale, v_scale   fp8 / int8 (either q type): per-cache dequantisation scales
 *                      (ignored for fp16 and bfloat16 caches) */
typedef struct {
  int32_t B, Hq, Hkv, D;
  int32_t block_size, num_blocks, max_blocks_per_seq;
  int32_t kv_dtype;
  float k_scale, v_scale;
} pd_dims;

/* Workspace bytes that decode_paged needs for these shapes, qlen and
 * num_splits (0 = balanced automatic split) on a device with sm_count SMs
 * (sm_count <= 0: the current device's). 0 means no workspace is needed (the
 * pointer may then be NULL). Layout: the fp32 split partials (m and l of
 * every partial row, then its O row); a split unit's pieces and their slots
 * follow from the sequence lengths, so nothing else is stored. Every
 * call writes what it later reads, so the buffer needs no initialisation and
 * one buffer serves any sequence of calls on one stream; calls that may run
 * at the same time must not share a workspace. Returns 0 for invalid dims. */
PD_API size_t pd_workspace_bytes(const pd_dims* dims, int qlen, int num_splits, int sm_count);

/* Number of CTAs decode_paged launches for these arguments (persistent grid),
 * or 0 for invalid dims. Host-only; no device work. */
PD_API int pd_grid_ctas(const pd_dims* dims, int qlen, int num_splits, int sm_count);

/* Paged decode attention, split-K over keys, GQA heads packed per CTA.
 * With a split (num_splits != 1) the call is two launches on `stream`: the
 * decode kernel, then a split-combine kernel launched with programmatic
 * dependent launch that merges the partials of units cut into pieces; a
 * fixed split of 2 to 16 pieces per unit whose pieces get one CTA each is
 * instead one launch of thread-block clusters (one per unit) that merge the
 * pieces themselves, when the device runs all those clusters at once.
 *
 *   q            fp16 [B*qlen, Hq, D] (bfloat16 for PD_KV_BF16, PD_KV_FP8_E4M3_BF16 and
 *                PD_KV_INT8_BF16); row b*qlen + i is query token i of sequence b
 *   k_cache      [num_blocks, block_size, Hkv, D] fp16, bfloat16, e4m3fn or int8
 *                (dims->kv_dtype)
 *   v_cache      same layout and dtype as k_cache
 *   block_table  int32 [B, max_blocks_per_seq]; entry [b][n] is the physical
 *                block holding keys n*block_size .. n*block_size+block_size-1 of
 *                sequence b. Only the entries of blocks holding visible keys are read.
 *   seq_lens     int32 [B]; keys cached for each sequence, query tokens included
 *   scale        multiplies q . k (e.g. 1/sqrt(D))
 *   window       sliding window in keys (<= 0: none)
 *   qlen         query tokens per sequence, 1..8; Hq/Hkv*qlen must be <= 32
 *   num_splits   0: balanced split of all visible key tiles over the SMs;
 *                >= 1: each sequence's visible tiles cut into num_splits
 *                contiguous chunks (1 = no split)
 *   out          q's type, [B*qlen, Hq, D], written in full (rows without a visible
 *                key are zeros); must not overlap the inputs
 *   workspace    device buffer of >= pd_workspace_bytes(...) bytes (contents need
 *                no initialisation; see pd_workspace_bytes)
 *   error_flag   device uint32 or NULL (see PD_DEVERR_*)
 *   stream       cudaStream_t to launch on
 * All pointers must be 16-byte aligned. */
PD_API pd_status decode_paged(const void* q, const void* k_cache, const void* v_cache,
                       const int32_t* block_table, const int32_t* seq_lens, float scale,
                       int window, int qlen, int num_splits, void* out, const pd_dims* dims,
                       void* workspace, size_t workspace_bytes, uint32_t* error_flag,
                       void* stream);

/* decode_paged with a different number of query tokens per sequence (the
 * multi-token verify cell of "Test Plan" generalised: a batch mixing plain
 * decode with speculative verify of varying depth).
 *   query_start_loc  device int32 [B+1], non-decreasing: sequence b owns rows
 *                    query_start_loc[b] .. query_start_loc[b+1]-1 of q and
 *                    out, its qlen_b = query_start_loc[b+1] - query_start_loc[b]
 *                    tokens at positions seq_lens[b] - qlen_b + i (i < qlen_b)
 *   num_query_tokens rows of q and out (total over the batch)
 *   max_qlen         an upper bound of every qlen_b, 1..8; it sizes the
 *                    kernel (G * max_qlen <= 32) and the workspace:
 *                    pd_workspace_bytes(dims, max_qlen, num_splits, 0)
 * Every other argument is decode_paged's. A sequence with qlen_b = 0 writes
 * nothing; rows of out outside [query_start_loc[0], query_start_loc[B]) are
 * not written. A range that decreases, exceeds max_qlen or leaves
 * [0, num_query_tokens) sets PD_DEVERR_QUERY_START and that sequence is
 * skipped. */
PD_API pd_status decode_paged_varlen(const void* q, const void* k_cache, const void* v_cache,
                                     const int32_t* block_table, const int32_t* seq_lens,
                                     const int32_t* query_start_loc, int num_query_tokens,
                                     int max_qlen, float scale, int window, int num_splits,
                                     void* out, const pd_dims* dims, void* workspace,
                                     size_t workspace_bytes, uint32_t* error_flag, void* stream);

/* Split-K combine on its own (the combine step of "Purpose" and of the
 * schedule model in "Test Result"). For each of `rows` rows and S partials:
 *   part_m  fp32 [rows, S]     largest score of the chunk, natural-log units
 *                              (-inf for an empty chunk)
 *   part_l  fp32 [rows, S]     sum over the chunk of exp(s_j - m)
 *   part_o  fp32 [rows, S, D]  sum over the chunk of exp(s_j - m) * V_j
 *   out     fp16 [rows, D]     sum_s w_s O_s / sum_s w_s l_s with
 *                              w_s = exp(m_s - max_s m_s); zeros when every
 *                              chunk is empty
 * D is 1..1024 and a multiple of 8. */
PD_API pd_status decode_paged_combine(const float* part_m, const float* part_l, const float* part_o,
                               int rows, int num_splits, int D, void* out, void* stream);

/* Paged KV-cache writer: stores the K and V rows of new tokens where the
 * decode reads them (opengfx1030/vllm-rdna pull request #33, "Test Plan": the
 * decode is checked against the paged writer's layout).
 *   k_new, v_new  fp16 [num_tokens, Hkv, D] (bfloat16 for PD_KV_BF16, PD_KV_FP8_E4M3_BF16
 *                 and PD_KV_INT8_BF16), 16-byte aligned
 *   slot_mapping  int64 [num_tokens], device; token t goes to block
 *                 slot / block_size, offset slot % block_size of both caches;
 *                 a negative slot is a padding token and writes nothing
 *   k_cache,      [num_blocks, block_size, Hkv, D] of dims->kv_dtype (16-byte
 *   v_cache       aligned for 16-bit kinds, 8-byte for one-byte codes), updated in place
 *   dims          Hkv, D (a multiple of 8), block_size, num_blocks, kv_dtype,
 *                 k_scale, v_scale are read; B, Hq, max_blocks_per_seq are not
 *   error_flag    device uint32 or NULL
 * fp16 and bfloat16 caches receive the input bits unchanged. fp8 / int8 caches receive the
 * code nearest to the IEEE fp32 quotient x / k_scale (V: v_scale): e4m3fn
 * with ties to even, saturating at +-448, NaN -> 0x7F; int8 with ties to even,
 * clamped to [-127, 127], NaN -> 0. A slot at or beyond num_blocks*block_size
 * writes nothing and sets PD_DEVERR_SLOT. Two tokens with the same slot race
 * (one of them wins). One launch on `stream`; nothing is allocated. */
PD_API pd_status write_kv_cache(const void* k_new, const void* v_new, const int64_t* slot_mapping,
                                int num_tokens, void* k_cache, void* v_cache, const pd_dims* dims,
                                uint32_t* error_flag, void* stream);

/* Failure-detection controls (process-wide, read at each launch; for tests of
 * the error path, not for production use).
 *   pd_set_wait_limit_ns: wall-time limit of every pipeline wait inside the
 *     decode kernel (0 restores the default, 2 s). A wait that runs past it
 *     sets PD_DEVERR_TIMEOUT; the kernel then skips its remaining waits and
 *     work, keeps its barrier sequence, lets every issued copy land and exits,
 *     so the CUDA context stays usable.
 *   pd_set_fault_injection: 1 makes the decode kernel's producer issue no
 *     loads, so the consumers' waits can only run out (a wait that nothing
 *     completes); 0 turns it off. The outputs of such calls are unspecified. */
PD_API void pd_set_wait_limit_ns(unsigned long long ns);
PD_API void pd_set_fault_injection(int mode);

/* Size of the scratch array built into the library for
 * decode_paged_static_scratch (32 MiB). Every GPU on which that entry point
 * has been called keeps this much device memory until the process exits. */
#define PD_STATIC_SCRATCH_BYTES (32u << 20)

/* decode_paged for callers that cannot allocate device memory (no counterpart
 * in the pages: it exists for this library's users). Some callers cannot call
 * cudaMalloc -- code running inside an allocator's own callbacks, a plugin
 * host that hands out no device buffers, a process whose device footprint is
 * fixed after start-up -- so they cannot provide decode_paged's workspace.
 * This entry point takes the same arguments minus the workspace and uses a
 * scratch array of PD_STATIC_SCRATCH_BYTES compiled into the library.
 *   - It allocates nothing: no cudaMalloc, no cudaFree, no allocating
 *     library routine. The caller still owns q, the caches, the tables,
 *     out and error_flag.
 *   - Calls whose workspace (pd_workspace_bytes) exceeds
 *     PD_STATIC_SCRATCH_BYTES return PD_ERR_WORKSPACE before anything runs.
 *   - Each call launches exactly as decode_paged does, on `stream`.
 *   - The first call on a device looks up the scratch's device address on
 *     that device (cudaGetSymbolAddress, the device being current). Under
 *     CUDA's lazy module loading (the default) that lookup is also when the
 *     driver loads the module holding the array and takes its
 *     PD_STATIC_SCRATCH_BYTES of device memory. So make the first call on
 *     each device at start-up: outside any allocator callback, while the
 *     process may still grow its footprint, and before any stream capture.
 *     Later calls take no device memory.
 *   - After a cudaDeviceReset the next call on that device is a first call
 *     again (the address is looked up in the new context).
 *   - All calls on a device share the one scratch array, which keeps the
 *     last call's contents: calls that may overlap on the GPU (different
 *     streams without ordering between them) race and give wrong results. */
PD_API pd_status decode_paged_static_scratch(const void* q, const void* k_cache, const void* v_cache,
                       const int32_t* block_table, const int32_t* seq_lens, float scale,
                       int window, int qlen, int num_splits, void* out, const pd_dims* dims,
                       uint32_t* error_flag, void* stream);

/* Human-readable name of a status. */
PD_API const char* pd_status_str(pd_status status);

#ifdef __cplusplus
}
#endif

#endif /* PDECODE_H */
