// Shared definitions of the libgdn kernels: launch parameters, the workspace
// layout and small device helpers. Nothing here computes the method itself.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/gdn.h"

namespace gdn {

constexpr int kChunk = 64;   // C: tokens per chunk
constexpr int kDk = 128;     // key head dimension
constexpr int kDv = 128;     // value head dimension

// Everything a kernel needs, passed by value. Pointers are device pointers.
struct Params {
  int T, N, H, Hv, HG, nt_max;
  int D;                     // head size of the tensors in memory (dk = dv; 64 or 128)
  const void* q;
  const void* k;
  const void* v;
  const float* g;
  const float* beta;
  float scale;
  const float* s0;           // [N, Hv, dv, dk] or null
  void* out;                 // [T, Hv, dv]
  float* sT;                 // [N, Hv, dv, dk] or null
  int32_t* status;           // device status word
  const int2* seq_info;      // [N] sanitized (start, length)
  const int32_t* chunk_offsets;  // [N + 1]
  const int2* chunk_table;   // [nt_max] (sequence, ordinal) or (-1, -1)
  const int32_t* seq_order;  // [N] the sequences longest first (the scan's launch order), or
                             // null for the given order
  float* G;                  // [nt_max, Hv, 64] in-chunk cumulative log-decay
  float* EF;                 // [nt_max, Hv, 128] exp(G) then exp(G_L - G) (tensor-core path,
                             // scalar gates)
  void* w;                   // [nt_max, Hv, 64, dk]
  float* u;                  // [nt_max, Hv, 64, dv]
  const int32_t* cu;         // cu_seqlens as given (or null), read only when early_one is set
  int pf_ahead;              // intra kernel: > 0 prefetches into L2 the tiles of the chunk
                             // slot this many ahead (about where the CTA that next takes its
                             // SM will be)
  int split_slots;           // intra kernel: the last split_slots chunk slots are each taken
                             // by two CTAs, one per half of the key head's value heads (the
                             // grid's last, partial wave in smaller pieces); 0 for none
  int early_one;             // one sequence whose chunk table this call builds: the intra
                             // kernel maps slot s to chunk s and requests its tiles before
                             // the table is written
  void* M;                   // [nt_max, Hv, 64, 64] (or hi/lo pair) decay-masked q.k
  void* k16;                 // fp16 images of the chunk's k tile (tensor-core path): per
                             // [nt_max, H] key head, or per [nt_max, Hv] value head with
                             // per-channel gates (the decay exp(G_L - G) applied)
  void* qimg;                // [nt_max, Hv] bf16 hi/lo images of exp(G) q (tensor-core path,
                             // per-channel gates)
  void* q16;                 // [nt_max, H] fp16 images of the chunk's q tile, 1/||q|| applied
                             // (tensor-core path, scalar gates)
  float* qt;                 // [nt_max, Hv, dk, 64] (exp(G) q)^T        (SIMT path)
  float* kt;                 // [nt_max, Hv, 64, dk] exp(G_L - G) k      (SIMT path)
  float* gam;                // [nt_max, Hv, dk] exp(G_L)                (SIMT path)
  float* hs;                 // [nt_max, Hv, dv, dk] chunk-start states, or null (backward)
  float* vn_out;             // [nt_max, Hv, 64, dv] v_new, or null (backward)
  const float* qrn;          // [T, H] 1/||q|| or null
  const float* krn;          // [T, H] 1/||k|| or null
  int out_bf16;
  uint32_t stall_polls;      // testing hook: > 0 makes the scan wait this many polls on an
                             // event that never happens (its timeout path); 0 normally
  int dbg_poison;            // testing hook of the GDN_DEBUG build (an out-of-range M slot)
  int m_f16;                 // tensor-core path: the M image as an fp16 hi/lo pair (the
                             // forward's scan), else a bf16 hi/lo pair (the backward's)
};

// Parameters of the backward kernels (device pointers; fp32 SIMT arithmetic). Per-slot
// arrays are indexed by slot = chunk slot * Hv + value head.
struct BwdParams {
  int T, N, H, Hv, HG, nt_max;
  const void* q;
  const void* k;
  const void* v;
  const float* g;
  const float* beta;
  float scale;
  const void* dout;          // [T, Hv, dv], bf16 when dout_bf16 else fp32
  int dout_bf16;
  const float* dfin;         // [N, Hv, dv, dk] gradient of the final state, or null
  float* dq;                 // [T, H, dk]
  float* dk;                 // [T, H, dk]
  float* dv;                 // [T, Hv, dv]
  float* dg;                 // [T, Hv]
  float* dbeta;              // [T, Hv]
  float* dh0;                // [N, Hv, dv, dk] gradient of the initial state, or null
  int32_t* status;
  const int2* seq_info;
  const int32_t* chunk_offsets;
  const int2* chunk_table;
  // forward quantities: the fp32 SIMT path's layout (fp32 inputs) ...
  const float* wT;           // [slot][D][64] w^T
  const float* kt;           // [slot][64][D] exp(G_L - G) k
  const float* qt;           // [slot][D][64] (exp(G) q)^T
  const float* MT;           // [slot][64][64] M^T
  const float* gam;          // [slot][D] exp(G_L)
  // ... or the tensor-core path's bridge (bf16 inputs)
  const void* wimg;          // [slot] bf16 w image (two swizzled [64][128 B] halves)
  const void* mimg;          // [slot] bf16 M hi/lo image ([128][128 B], swizzled)
  const float* G;            // [slot][64] in-chunk cumulative gate
  const float* hs;           // [slot][D][D] chunk-start state, [dv][dk]
  const float* vn;           // [slot][64][D] v_new
  // backward intermediates
  float* dvn;                // [slot][64][D] gradient of v_new
  float* dhs;                // [slot][D][D] gradient of the next chunk-start state, [dv][dk]
  float* dos;                // [slot][64][D] dO S^T
  float* dw;                 // [slot][64][D] gradient of w: -dv_new S^T
  float* ys;                 // [slot][64][D] v_new dS_next^T
  float* sdot;               // [slot] <S, dS_next>
  float* ttdw;               // [slot][64][D] T^T dw
  float* dqp;                // [slot][64][D] this value head's part of dq
  float* dkp;                // [slot][64][D] this value head's part of dk
};

// Parameters of the token-serial kernel (device pointers).
struct RecParams {
  int T, N, H, Hv, HG;
  const void* q;
  const void* k;
  const void* v;
  const float* g;
  const float* beta;
  float scale, eps;
  const float* s0;      // [N, Hv, dv, dk] or null
  void* out;            // [T, Hv, dv]
  float* sT;            // [N, Hv, dv, dk] or null
  const int32_t* cu;    // [N + 1] or null (one sequence of T rows)
  int32_t* status;      // device status word or null
  int bf16_in, out_bf16, l2norm;
};

// Parameters of the front-end kernels (device pointers).
struct ConvParams {
  int T, N, H, Hv, C, d, n_snap;
  const void* x;        // [T, C] projection output (q | k | v channels)
  const float* w;       // [C, d] conv taps
  const float* s_in;    // [N, C, d - 1] or null (zeros)
  float* s_out;         // [N, C, d - 1] or null
  float* snaps;         // [N, n_snap, C, d - 1] or null
  void* q;              // [T, H, dk]
  void* k;              // [T, H, dk]
  void* v;              // [T, Hv, dv]
  const int32_t* cu;    // [N + 1] or null
  int32_t* status;      // device status word or null
  float eps;
  int bf16, l2norm;
};

// Byte offsets of the workspace regions (each 256-byte aligned), and the extent
// [begin, end) of every region in order (for the guard-band check of the tests).
struct WsLayout {
  size_t status, seq_info, chunk_offsets, chunk_table, seq_order, G, EF, w, u, M, k16, qimg,
      q16, qt, kt, gam, qrn, krn, total;
  static constexpr int kMaxRegions = 16;
  int nreg;
  size_t rbeg[kMaxRegions], rend[kMaxRegions];
};

__host__ __device__ inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Layout for a problem with head size D. The tensor-core path stores w in bf16, M as
// a hi/lo bf16 pair and the in-chunk gate sums G, always at head size 128 (a head of
// 64 runs zero-padded to 128: the tensor maps fill the missing half with zeros); the
// fp32 SIMT path stores w^T, u, M^T and the decayed q / k images and exp(G_L) in fp32.
// `guard` bytes are left free after every region (GDN_FLAG_WORKSPACE_GUARDS).
inline WsLayout ws_layout(int T, int N, int H, int Hv, int nt_max, bool tc_path, bool l2norm,
                          int D = kDk, bool channel_gates = false, size_t guard = 0) {
  WsLayout L{};
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    if (L.nreg < WsLayout::kMaxRegions) {
      L.rbeg[L.nreg] = at;
      L.rend[L.nreg] = at + bytes;
      ++L.nreg;
    }
    o = align_up(o + bytes, 256) + guard;
    return at;
  };
  L.status = take(64);
  L.seq_info = take(sizeof(int2) * (size_t)N);
  L.chunk_offsets = take(sizeof(int32_t) * (size_t)(N + 1));
  L.chunk_table = take(sizeof(int2) * (size_t)nt_max);
  L.seq_order = take(sizeof(int32_t) * (size_t)N);
  const size_t slots = (size_t)nt_max * (size_t)Hv;
  L.G = tc_path ? take(sizeof(float) * slots * kChunk) : 0;
  L.EF = (tc_path && !channel_gates) ? take(sizeof(float) * slots * 2 * kChunk) : 0;
  const size_t Dw = tc_path ? kDk : D;
  L.w = take((tc_path ? 2 : 4) * slots * kChunk * Dw);
  L.u = take(sizeof(float) * slots * kChunk * Dw);
  L.M = take(4 * slots * kChunk * kChunk);
  const bool tc_ch = tc_path && channel_gates;  // per value head k images, q images, exp(G_L)
  L.k16 = tc_path ? take((size_t)nt_max * (tc_ch ? Hv : H) * kChunk * kDk * 2) : 0;
  L.qimg = tc_ch ? take(slots * 2 * kChunk * kDk * 2) : 0;
  L.q16 = (tc_path && !channel_gates) ? take((size_t)nt_max * H * kChunk * kDk * 2) : 0;
  L.qt = tc_path ? 0 : take(sizeof(float) * slots * kChunk * D);
  L.kt = tc_path ? 0 : take(sizeof(float) * slots * kChunk * D);
  L.gam = tc_path ? (tc_ch ? take(sizeof(float) * slots * kDk) : 0)
                  : take(sizeof(float) * slots * D);
  L.qrn = l2norm ? take(sizeof(float) * (size_t)T * H) : 0;
  L.krn = l2norm ? take(sizeof(float) * (size_t)T * H) : 0;
  L.total = o;
  return L;
}

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

// Programmatic dependent launch: a kernel launched with the programmatic-serialization
// attribute may start before its predecessor in the stream has finished; pdl_wait()
// blocks until the predecessor has completed and its writes are visible (a no-op for
// a kernel launched without the attribute); pdl_release() lets the successor start.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }
__device__ __forceinline__ void pdl_release() {
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
}

__device__ __forceinline__ void set_status(int32_t* status, int bits) {
  if (status) atomicOr(status, bits);
}

// Device-side index check of the GDN_DEBUG build: returns whether an index that
// addresses global memory is in its range, raising GDN_DEV_DEBUG_INDEX when it is not (the
// caller then skips or redirects the access). Always true, and free, in the normal build.
__device__ __forceinline__ bool dbg_ok(bool in_range, int32_t* status) {
#ifdef GDN_DEBUG
  if (!in_range) set_status(status, GDN_DEV_DEBUG_INDEX);
  return in_range;
#else
  (void)in_range;
  (void)status;
  return true;
#endif
}

// The (start, length) of sequence n and its first chunk slot.
struct SeqView {
  int start, len, first_slot;
};

template <typename P>
__device__ __forceinline__ SeqView seq_view(const P& p, int n) {
  int2 si = p.seq_info[n];
  return SeqView{si.x, si.y, p.chunk_offsets[n]};
}

// Testing hook (gdn_test_scan_timeout): polls of the scan's never-completing wait for the
// next launches, 0 normally.
uint32_t scan_stall_polls();
// Testing hook of the GDN_DEBUG build (gdn_test_debug_poison), 0 normally.
int debug_poison();

// Raise a kernel's dynamic shared-memory limit once per (kernel, device), so
// that later calls (for example under CUDA-graph capture) make no attribute call.
void ensure_smem_limit(const void* kernel, int bytes);

// Launch `kernel` on `s` with the programmatic-serialization attribute (see pdl_wait).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t s, Args&&... args) {
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

// Kernel launchers (one translation unit each).
// Sequence counts up to which the chunk-table kernel also writes the longest-first order.
constexpr int kMaxOrderedSeqs = 1024;
void launch_chunk_table(const int32_t* cu, int N, int T, int nt_max, int2* table,
                        int32_t* offsets, int2* seq_info, int32_t* status, cudaStream_t s,
                        bool zero_status = false, int32_t* seq_order = nullptr);
void launch_l2norm(const void* q, const void* k, bool bf16, int T, int H, int D, float eps,
                   float* qrn, float* krn, cudaStream_t s);
bool launch_gen_intra(const Params& p, int D, bool channel_gates, bool bf16_inputs, cudaStream_t s);
bool launch_gen_inter(const Params& p, int D, cudaStream_t s);
// ev: null, or three events recorded after the reverse scan, after the contractions with
// the stored states and after the per-chunk gradient kernels.
// tc_bridge: the forward quantities are the tensor-core path's bridge (bf16 inputs).
bool launch_bwd(const BwdParams& p, int D, bool bf16_inputs, bool tc_bridge, cudaStream_t s,
                cudaEvent_t* ev);
bool launch_bwd_scan_tc(const BwdParams& p, int D, cudaStream_t s);
bool launch_tc_intra(const Params& p, cudaStream_t s);
bool launch_tc_inter(const Params& p, bool channel_gates, cudaStream_t s);
// The scalar-gate scan (k_scan.cu); launch_tc_inter routes scalar gates to it.
bool launch_scan(const Params& p, cudaStream_t s);
bool launch_kda_intra(const Params& p, cudaStream_t s);
bool launch_recurrent(const RecParams& p, cudaStream_t s);
bool launch_conv_front(const ConvParams& p, cudaStream_t s);

// Encode a TMA tensor map over a bf16 [rows, heads, 128] tensor with a box of
// 64 rows x 1 head x 64 elements and the 128-byte swizzle. False on failure.
bool encode_rows_tmap(void* tmap, const void* base, int rows, int heads, int D);
// Plain 2-D tensor map over a row-major [rows, cols] bf16 or fp32 matrix (no swizzle).
bool encode_2d_tmap(void* tmap, const void* base, bool bf16, int cols, int rows, int box_cols,
                    int box_rows);
// Same over an fp32 state [rows, 128]: box 32 rows x 32 elements, 128-byte swizzle.
bool encode_state_tmap(void* tmap, const float* base, int rows);

}  // namespace gdn
