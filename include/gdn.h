/*
 * gdn.h -- C ABI of libgdn: the chunked gated-delta-rule prefill forward
 * on one NVIDIA GB300 (sm_103a).
 *
 * The operation (per sequence n, value head hv, key head h = hv / (Hv / H);
 * the per-head fp32 state S has one row per key dimension):
 *
 *   S_t = exp(g_t) * S_{t-1} + beta_t * k_t (v_t - exp(g_t) * S_{t-1}^T k_t)^T
 *   o_t = scale * S_t^T q_t
 *
 * evaluated in chunks of C = 64 tokens: an intra-chunk stage parallel over
 * [chunks, key heads] and an inter-chunk scan parallel over [sequences, value
 * heads], the two-stage split of "Optimizing GDN Chunk Prefill on Intel AMX
 * CPU" (sections 3-5). The per-token update is the one described in
 * "Chunking Qwen3.5's gated DeltaNet for 1.5x faster prefill on Apple
 * Silicon" (section "What is the gated delta rule in Qwen3.5?"). Varlen
 * packing via cu_seqlens and the static [NT_max, 2] chunk table with
 * sentinel slots follow the FLA RFC "Graph capture support for prefill and
 * training" (section "Core design").
 *
 * Conventions for every entry point:
 *   - All tensor pointers are DEVICE pointers owned by the caller. The library
 *     never allocates, frees or synchronizes; it enqueues work on `stream` and
 *     returns. Nothing is read back to the host, so a call can be captured in
 *     a CUDA graph (addresses are then fixed by the caller).
 *   - Layouts are dense, row-major, innermost dimension last:
 *       q, k            [T, H, dk]   (gdn_desc.qkv_dtype)
 *       v               [T, Hv, dv]  (gdn_desc.qkv_dtype)
 *       out             [T, Hv, dv]  (gdn_desc.out_dtype)
 *       g, beta         [T, Hv]      fp32; g is the per-token log-decay (<= 0)
 *                       (g is [T, Hv, dk] with GDN_FLAG_CHANNEL_GATES: one
 *                       log-decay per key channel, decaying that row of S)
 *       states          [N, Hv, dv, dk] fp32 (value-major, "[N, Hv, V, K]")
 *       cu_seqlens      [N + 1] int32 prefix sums of sequence lengths
 *       chunk_indices   [nt_max, 2] int32 (sequence id, chunk ordinal)
 *       chunk_offsets   [N + 1] int32 (first slot of each sequence; [N] = total)
 *   - Return value: GDN_OK (0) or a negative gdn_status. On an argument error
 *     nothing is enqueued. Problems that only the data reveals (malformed
 *     cu_seqlens, more chunks than nt_max, a bad caller-supplied chunk table)
 *     never fault: the kernels clamp or skip and set bits of the device status
 *     word (gdn_dev_status), which gdn_read_status copies back.
 *   - Supported: dk = dv = 128 or dk = dv = 64 (the head sizes of "Optimizing
 *     GDN Chunk Prefill on Intel AMX CPU", section 9), chunk_size = 64,
 *     Hv % H == 0, scalar or per-channel gates. bf16 inputs with dk = 128 and
 *     scalar gates run on the tensor-core kernels; every other case runs on the
 *     fp32 SIMT kernels of the same intra/inter split. gdn_recurrent_fwd and
 *     gdn_conv_front take dk = dv = 128 and scalar gates only.
 */
#ifndef GDN_H_
#define GDN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same definitions as the CUDA runtime's, so that this header stands alone. */
typedef struct CUstream_st* cudaStream_t;
typedef struct CUevent_st* cudaEvent_t;

typedef enum gdn_dtype { GDN_F32 = 0, GDN_BF16 = 1 } gdn_dtype;

typedef enum gdn_status {
  GDN_OK = 0,
  GDN_ERR_NULL_ARG = -1,          /* a required pointer is NULL */
  GDN_ERR_BAD_SHAPE = -2,         /* T < 0, N < 1, H < 1, Hv % H != 0, nt_max < 0 */
  GDN_ERR_UNSUPPORTED = -3,       /* valid but not built: head size, chunk_size != 64, dtype, flag */
  GDN_ERR_MISALIGNED = -4,        /* a pointer is not 16-byte aligned (workspace: 256 bytes) */
  GDN_ERR_WORKSPACE_TOO_SMALL = -5,
  GDN_ERR_LAUNCH_FAILED = -6      /* the CUDA runtime refused a launch or copy */
} gdn_status;

/* Bits of the device status word (OR-ed by the kernels, cleared per call). */
typedef enum gdn_dev_status {
  GDN_DEV_BAD_CU_SEQLENS = 1,     /* cu_seqlens not monotone or beyond T: clamped */
  GDN_DEV_CHUNK_OVERFLOW = 2,     /* more chunks than nt_max: the excess is skipped */
  GDN_DEV_BAD_CHUNK_TABLE = 4,    /* caller table names a chunk that does not exist: skipped;
                                     also set if the table built for one sequence disagrees
                                     with the slot = chunk mapping the intra kernel assumes
                                     when it requests its tiles early (an internal error) */
  GDN_DEV_TIMEOUT = 8,            /* a bounded on-chip wait gave up (results invalid) */
  GDN_DEV_NONFINITE = 16,         /* a state or output of the bf16 tensor-core path came out
                                     non-finite: an fp16 operand (state, decayed v_new) left
                                     the fp16 range, or the inputs held inf/NaN */
  GDN_DEV_DEBUG_INDEX = 32        /* (GDN_DEBUG builds only) an index that addresses global
                                     memory in the chunk-table, intra or scan kernel was out of
                                     its range: that access was skipped or redirected */
} gdn_dev_status;

enum {
  GDN_FLAG_QK_L2NORM = 1u,            /* normalise q and k rows: x / sqrt(sum x^2 + eps) */
  GDN_FLAG_BUILD_CHUNK_INDICES = 2u,  /* fill the caller's chunk_indices buffer */
  GDN_FLAG_CHANNEL_GATES = 4u,        /* g is [T, Hv, dk]: a gate per key channel */
  GDN_FLAG_WORKSPACE_GUARDS = 8u      /* leave a 4 KiB gap after every workspace region
                                         (a caller may fill the workspace with a pattern
                                         and check the gaps after the call; see
                                         gdn_workspace_regions); results are unchanged */
};

enum { GDN_NUM_STAGE_EVENTS = 5 };

/*
 * Problem descriptor (plain data; the pages' Python signature infers these
 * from tensor shapes). Fields:
 *   T            rows of q, k, v, g, beta, out (the token budget T_max when the
 *                call is graph-captured; rows past cu_seqlens[N] are ignored and
 *                their out rows are left untouched)
 *   N            number of sequences (cu_seqlens has N + 1 entries; zero-length
 *                sequences are allowed, e.g. padding up to N_max)
 *   H, Hv        key/query heads and value heads; Hv must be a multiple of H
 *   dk, dv       head dimensions: dk = dv = 128 or dk = dv = 64
 *   chunk_size   64
 *   nt_max       number of chunk slots; 0 selects cdiv(T, 64) + N - 1, which
 *                bounds the chunk count of any cu_seqlens with N sequences
 *                and at most T tokens
 *   qkv_dtype    gdn_dtype of q, k, v; out_dtype: gdn_dtype of out
 *   flags        GDN_FLAG_* bits
 *   l2norm_eps   eps of the optional L2 norm; <= 0 selects 1e-6
 *   workspace    device scratch of at least gdn_workspace_size(desc) bytes,
 *                256-byte aligned, owned by the caller; it must not be used by
 *                another call that may run at the same time
 *   stage_events NULL, or an array of GDN_NUM_STAGE_EVENTS cudaEvent_t that
 *                gdn_chunk_fwd records on `stream` before the first kernel and
 *                after the chunk-table, intra-chunk and inter-chunk kernels (the
 *                first four; gdn_chunk_bwd records all five), for timing each
 *                stage; the library does not create them
 */
typedef struct gdn_desc {
  int32_t T;
  int32_t N;
  int32_t H;
  int32_t Hv;
  int32_t dk;
  int32_t dv;
  int32_t chunk_size;
  int32_t nt_max;
  int32_t qkv_dtype;
  int32_t out_dtype;
  uint32_t flags;
  float l2norm_eps;
  void* workspace;
  size_t workspace_bytes;
  cudaEvent_t* stage_events;
} gdn_desc;

/*
 * Validate a descriptor's dimensions, dtypes and flags (host only; pointers
 * other than the workspace are not looked at). Returns GDN_OK or the status
 * gdn_chunk_fwd would return for it.
 */
int gdn_check_desc(const gdn_desc* desc);

/*
 * The chunk-slot bound nt_max = cdiv(T, chunk_size) + N - 1 of the FLA RFC
 * ("Core design": the first sequence's partial chunk is covered by the cdiv
 * term, every further sequence adds at most one). Returns -1 for T < 0 or N < 1.
 */
int32_t gdn_nt_max(int32_t T, int32_t N, int32_t chunk_size);

/*
 * Bytes of workspace gdn_chunk_fwd needs for this descriptor (the fields
 * workspace and workspace_bytes are ignored). 0 if the descriptor is invalid.
 * Size follows the static bound: it depends on T, N, nt_max, H, Hv and dtypes,
 * not on the contents of cu_seqlens.
 */
size_t gdn_workspace_size(const gdn_desc* desc);

/*
 * Device-side chunk-index builder (FLA RFC, "Core design": a searchsorted
 * routine fills a fixed [NT_max, 2] table and marks unused slots with a
 * sentinel). For every slot s < nt_max it writes (n, c): the sequence n whose
 * chunks cover slot s and the chunk ordinal c inside it (token start =
 * cu_seqlens[n] + 64 c), slots ordered by sequence and then ordinal, and
 * (-1, -1) in unused slots. chunk_offsets[n] receives the slot of sequence n's
 * first chunk and chunk_offsets[N] the total number of chunks.
 *   cu_seqlens     [N + 1] int32, or NULL for one sequence of T tokens
 *   chunk_indices  [nt_max, 2] int32 output, or NULL to skip the table
 *   chunk_offsets  [N + 1] int32 output (required)
 *   status         one int32 of device memory the kernel ORs gdn_dev_status
 *                  bits into (not cleared here), or NULL
 * Malformed cu_seqlens are clamped to [0, T] and made monotone (status bit 1);
 * chunks beyond nt_max are not written (status bit 2).
 */
int gdn_build_chunk_indices(const int32_t* cu_seqlens, int32_t N, int32_t T,
                            int32_t nt_max, int32_t* chunk_indices,
                            int32_t* chunk_offsets, int32_t* status,
                            cudaStream_t stream);

/*
 * The chunked gated-delta-rule forward (the whole hot path: optional q/k
 * L2-norm prologue, chunk-table builder, intra-chunk kernel, inter-chunk scan).
 *   q, k, v        inputs (layouts above), dtype desc->qkv_dtype
 *   g, beta        fp32 [T, Hv] (g: [T, Hv, dk] with GDN_FLAG_CHANNEL_GATES)
 *   scale          output scale; <= 0 or NaN selects 1/sqrt(dk)
 *   initial_state  fp32 [N, Hv, dv, dk] or NULL for zeros
 *   cu_seqlens     int32 [N + 1] or NULL for one sequence of T tokens (N = 1)
 *   chunk_indices  NULL: the table is built inside the workspace;
 *                  non-NULL and GDN_FLAG_BUILD_CHUNK_INDICES set: the table is
 *                  built into this caller buffer [nt_max, 2];
 *                  non-NULL without the flag: the caller's table is read (it
 *                  must list every real chunk once; sentinel rows are skipped)
 *   out            [T, Hv, dv], dtype desc->out_dtype; rows outside the
 *                  sequences are not written
 *   final_state    fp32 [N, Hv, dv, dk] or NULL (not written). It may alias
 *                  initial_state: each slice is read before it is written.
 *                  A zero-length sequence gets its initial state (or zeros).
 * Rows of a partial last chunk are masked (beta = 0, k = 0, g = 0 past the end
 * of the sequence) and never stored.
 */
int gdn_chunk_fwd(const gdn_desc* desc, const void* q, const void* k,
                  const void* v, const float* g, const float* beta, float scale,
                  const float* initial_state, const int32_t* cu_seqlens,
                  int32_t* chunk_indices, void* out, float* final_state,
                  cudaStream_t stream);

/*
 * Workspace bytes gdn_chunk_bwd needs for this descriptor (0 if the descriptor
 * is invalid or not supported by the backward pass).
 */
size_t gdn_bwd_workspace_size(const gdn_desc* desc);

/*
 * The backward pass of gdn_chunk_fwd (scalar gates; no q/k L2 norm): given the
 * gradient of a loss with respect to out (d_out) and to final_state
 * (d_final_state, NULL for none), the gradients with respect to q, k, v, g,
 * beta and initial_state. It is the chunked form of the recurrence's adjoint,
 * run as the backward kernels the FLA graph-capture RFC lists for GDN ("What
 * needs to change": the state-gradient scan, the local dv, dq/dk/dw/dg and
 * WY-representation gradients): a forward recompute that keeps each chunk's
 * start state and v_new, a reverse scan over the chunks for the state
 * gradient, and per-chunk kernels for the rest, all in fp32 arithmetic.
 *   q, k, v, g, beta, scale, initial_state, cu_seqlens, chunk_indices
 *                  as for gdn_chunk_fwd (the same values as the forward call)
 *   d_out          [T, Hv, dv] in desc->out_dtype
 *   d_final_state  fp32 [N, Hv, dv, dk] or NULL (zero)
 *   dq, dk         fp32 [T, H, dk] (summed over the value heads of each key head)
 *   dv             fp32 [T, Hv, dv]
 *   dg, dbeta      fp32 [T, Hv]
 *   d_initial_state fp32 [N, Hv, dv, dk] or NULL (not written)
 * Rows outside the sequences are not written. desc->workspace must hold
 * gdn_bwd_workspace_size(desc) bytes. desc->stage_events, when set, are recorded
 * before the forward recompute and after it, after the reverse scan, after the
 * contractions with the stored states and after the per-chunk gradient kernels. Errors: as gdn_chunk_fwd, plus
 * GDN_ERR_UNSUPPORTED for GDN_FLAG_CHANNEL_GATES or GDN_FLAG_QK_L2NORM.
 */
int gdn_chunk_bwd(const gdn_desc* desc, const void* q, const void* k, const void* v,
                  const float* g, const float* beta, float scale,
                  const float* initial_state, const int32_t* cu_seqlens,
                  int32_t* chunk_indices, const void* d_out, const float* d_final_state,
                  float* dq, float* dk, float* dv, float* dg, float* dbeta,
                  float* d_initial_state, cudaStream_t stream);

/*
 * Host-only description of the workspace layout for this descriptor (as
 * gdn_workspace_size computes it): writes the byte range [begin[i], end[i]) of
 * each region the library may write, in increasing order, for the first
 * max_regions regions, and returns the number of regions (at most 16), or a
 * negative gdn_status for an invalid descriptor. Bytes of the workspace outside
 * every region are never written, so with GDN_FLAG_WORKSPACE_GUARDS the 4 KiB gap
 * after each region is a guard band a test can fill and check (the device-side
 * substitute for an out-of-bounds checker). The layout has no counterpart in the
 * pages.
 */
int gdn_workspace_regions(const gdn_desc* desc, size_t* begin, size_t* end, int max_regions);

/*
 * Enqueue an asynchronous copy of the device status word of the last call
 * that used desc->workspace into *host_status (pinned host memory is best).
 * The caller synchronizes the stream before reading it.
 */
int gdn_read_status(const gdn_desc* desc, int32_t* host_status, cudaStream_t stream);

/*
 * Size of the scratch array gdn_chunk_fwd_noalloc uses in place of a
 * workspace (64 MiB, held on every GPU that loads the library until exit).
 */
enum { GDN_NOALLOC_SCRATCH_BYTES = 64 << 20 };

/*
 * gdn_chunk_fwd without a workspace, for callers that may not allocate device
 * memory themselves (a framework that owns all device memory through its own
 * arena, or a serving loop that cannot afford an allocation's device
 * synchronization). The pages have no counterpart: this is a convenience of
 * this library. Same arguments and results as gdn_chunk_fwd; desc->workspace
 * and desc->workspace_bytes are ignored. The scratch is one file-scope device
 * array of GDN_NOALLOC_SCRATCH_BYTES shared by every call in the process:
 *   - a problem whose gdn_workspace_size exceeds it is rejected with
 *     GDN_ERR_WORKSPACE_TOO_SMALL and nothing is enqueued (T = 1024 with
 *     Hv = 32 fits; T = 4096 with Hv = 32 does not);
 *   - calls that may overlap on the GPU (other streams or host threads) race
 *     on the array: the caller must order them;
 *   - every call looks up the array's device address on the current device
 *     (cudaGetSymbolAddress; nothing is cached, so a device reset leaves no
 *     stale address); the first lookup on a device may load the library's
 *     device code, so make the first call outside stream capture;
 *   - the kernels' device status word (gdn_dev_status bits) lives in the
 *     array: read the last call's with gdn_noalloc_read_status, not
 *     gdn_read_status (which needs desc->workspace).
 * It calls no allocator (no cudaMalloc, cudaFree or library allocation).
 */
int gdn_chunk_fwd_noalloc(const gdn_desc* desc, const void* q, const void* k,
                          const void* v, const float* g, const float* beta, float scale,
                          const float* initial_state, const int32_t* cu_seqlens,
                          int32_t* chunk_indices, void* out, float* final_state,
                          cudaStream_t stream);

/*
 * Enqueue an asynchronous copy of the device status word of the last
 * gdn_chunk_fwd_noalloc call on the current device (the one in the shared
 * scratch array) into *host_status. Like the entry point it belongs to, it has
 * no counterpart in the pages. The caller synchronizes the stream before
 * reading *host_status; a call still running on another stream would race.
 * GDN_ERR_NULL_ARG for a NULL host_status, GDN_ERR_LAUNCH_FAILED if the copy
 * could not be enqueued.
 */
int gdn_noalloc_read_status(int32_t* host_status, cudaStream_t stream);

/*
 * Token-serial forward of the same recurrence, for decode (one token per
 * sequence) and speculative verification (a few tokens per sequence):
 * "Chunking Qwen3.5's gated DeltaNet for 1.5x faster prefill on Apple Silicon",
 * sections "How does decode run a sequential update on a GPU?" (one thread per
 * value column of a head's fp32 state, held on chip for the whole call) and
 * "Does the chunked kernel match the serial one?" (verification reproduces
 * decode's numerics). Per token: decay exp(g), the state's prediction for k,
 * the rank-1 correction with beta, then o = scale * S^T q (q and k
 * L2-normalised first when GDN_FLAG_QK_L2NORM is set).
 *
 * Guarantee: a call over n tokens of a sequence performs, token by token, the
 * same fp32 operations as n calls over one token each with the state passed
 * along (final_state of one call as initial_state of the next), so outputs and
 * states agree bit for bit.
 *
 * Arguments, layouts and ownership as gdn_chunk_fwd (q, k [T,H,dk]; v, out
 * [T,Hv,dv]; g, beta fp32 [T,Hv]; states fp32 [N,Hv,dv,dk]; cu_seqlens int32
 * [N+1] or NULL for one sequence of T rows; final_state may alias
 * initial_state; either may be NULL). The descriptor is validated as for
 * gdn_chunk_fwd, and dk = dv = 128 with scalar gates is required
 * (GDN_ERR_UNSUPPORTED otherwise); chunk_size, nt_max and the other flags
 * play no part. No workspace is needed: when desc->workspace is non-NULL its
 * status word is cleared and receives GDN_DEV_BAD_CU_SEQLENS for a malformed
 * cu_seqlens (clamped to [0, T]; a decreasing pair is an empty sequence), as
 * gdn_read_status reports. Work grows linearly with the tokens of a sequence:
 * long prompts belong to gdn_chunk_fwd. Errors: negative gdn_status before
 * anything is enqueued (NULL q/k/v/g/beta/out, bad shape, misalignment: 16
 * bytes for the tensors), GDN_ERR_LAUNCH_FAILED after a failed launch.
 */
int gdn_recurrent_fwd(const gdn_desc* desc, const void* q, const void* k, const void* v,
                      const float* g, const float* beta, float scale,
                      const float* initial_state, const int32_t* cu_seqlens, void* out,
                      float* final_state, cudaStream_t stream);

/*
 * Front end: the qkv projection output of a gated-DeltaNet layer to q, k, v
 * (the llama.cpp page, PrismML-Eng/llama.cpp pull 399, "What", item 1, and "How
 * (exactness)"): per channel a causal depthwise convolution of width d_conv whose
 * inputs are the d_conv - 1 inputs saved from before the sequence (the conv
 * state) followed by the sequence's rows, summed in tap order
 * (sum += w[j] * xx[t + j], j = 0 .. d_conv - 1, fp32, no bias), then SiLU, then,
 * when GDN_FLAG_QK_L2NORM is set, each q and k head row divided by
 * sqrt(sum x^2 + eps) (for gdn_chunk_fwd prefer leaving the flag off here and
 * setting it there, where the norm stays an fp32 factor instead of a rounded copy).
 *
 *   x               [T, C] in desc->qkv_dtype, C = 2*H*dk + Hv*dv, channels q | k | v
 *   conv_w          fp32 [C, d_conv], 1 <= d_conv <= 8
 *   conv_state_in   fp32 [N, C, d_conv - 1] (oldest first) or NULL for zeros
 *   cu_seqlens      int32 [N + 1] or NULL (one sequence of T rows); rows outside
 *                   every sequence are not written
 *   q, k            [T, H, dk]; v [T, Hv, dv]; desc->qkv_dtype (the x dtype)
 *   conv_state_out  fp32 [N, C, d_conv - 1] or NULL: the last d_conv - 1 inputs of
 *                   each sequence (old state entries when it is shorter); may alias
 *                   conv_state_in
 *   snapshots       fp32 [N, n_snapshots, C, d_conv - 1] or NULL: row s is the state
 *                   after the sequence's token s (after its last token for s past
 *                   the end), for rolling a speculative batch back; must not alias
 *                   conv_state_in
 *
 * The descriptor is validated as for gdn_chunk_fwd, and dk = dv = 128 is
 * required (GDN_ERR_UNSUPPORTED otherwise; chunk_size, nt_max, out_dtype and
 * GDN_FLAG_CHANNEL_GATES play no part). desc->workspace, when non-NULL, receives the status
 * word (GDN_DEV_BAD_CU_SEQLENS for a malformed cu_seqlens, clamped to [0, T]).
 * Errors: negative gdn_status before anything is enqueued (NULL x/conv_w/q/k/v,
 * bad d_conv or n_snapshots, misalignment: 16 bytes for x, q, k, v),
 * GDN_ERR_LAUNCH_FAILED after a failed launch.
 */
int gdn_conv_front(const gdn_desc* desc, const void* x, const float* conv_w, int32_t d_conv,
                   const float* conv_state_in, const int32_t* cu_seqlens, void* q, void* k,
                   void* v, float* conv_state_out, float* snapshots, int32_t n_snapshots,
                   cudaStream_t stream);

/*
 * Testing hook (no counterpart in the pages). With polls > 0, the bf16 scan of
 * the calls that follow (on any thread) first waits, for at most `polls`
 * polls, on an on-chip event that never happens; the wait runs out and the scan
 * takes its timeout path: GDN_DEV_TIMEOUT in the status word, every warp runs on
 * without waiting, the results of that call are invalid, and every copy in
 * flight is still waited for (at the full bound) before the kernel ends, so the
 * device stays usable. polls = 0 (the default) turns it off. It lets a test
 * exercise that path without a fault or a hang.
 */
void gdn_test_scan_timeout(uint32_t polls);

/*
 * 1 when this library was compiled with GDN_DEBUG (libgdn_debug.so), else 0.
 * The GDN_DEBUG build checks, in the device code of the chunk-table, intra and
 * scan kernels, every index that addresses a global-memory copy or store of
 * the bf16 forward path (chunk slot, key and value head, token row) against
 * its range before the access; an index out of range sets
 * GDN_DEV_DEBUG_INDEX and the access is skipped (a load is redirected to the
 * region's first slot so that its transaction count still completes).
 */
int gdn_debug_build(void);

/*
 * Testing hook for the GDN_DEBUG build (no counterpart in the pages; the
 * normal build ignores it). With on != 0, in the calls that follow the intra
 * kernel's CTA of chunk slot 0 and key head 0 aims its M image copies at value
 * slot nt_max * Hv, one past the end of the M region (inside the workspace,
 * whose next region follows): the device check must catch it, skip the copies
 * and set GDN_DEV_DEBUG_INDEX. on = 0 (the default) turns it off.
 */
void gdn_test_debug_poison(int32_t on);

/* Static description of a gdn_status value. */
const char* gdn_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* GDN_H_ */
