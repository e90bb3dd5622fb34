// Host side of the libgdn C ABI (include/gdn.h): argument validation,
// workspace carve-up and the launch sequence. No allocation, no
// synchronization, no device reads: every call only enqueues on `stream`.
#include <math.h>

#include <cuda.h>

#include <atomic>
#include <map>
#include <mutex>
#include <utility>

#include "gdn_common.cuh"

using namespace gdn;

namespace gdn {

namespace {
std::atomic<uint32_t> g_scan_stall_polls{0};
}  // namespace

uint32_t scan_stall_polls() { return g_scan_stall_polls.load(std::memory_order_relaxed); }
std::atomic<int> g_debug_poison{0};
int debug_poison() { return g_debug_poison.load(std::memory_order_relaxed); }

void ensure_smem_limit(const void* kernel, int bytes) {
  // largest limit set so far per (kernel, device); raised when a call needs more
  static std::mutex mu;
  static std::map<std::pair<const void*, int>, int> done;
  int dev = 0;
  cudaGetDevice(&dev);
  std::lock_guard<std::mutex> lock(mu);
  auto it = done.find({kernel, dev});
  if (it != done.end() && it->second >= bytes) return;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) ==
      cudaSuccess)
    done[{kernel, dev}] = bytes;
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// cuTensorMapEncodeTiled through the runtime's driver entry point (no libcuda link).
static EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = []() -> EncodeTiledFn {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<EncodeTiledFn>(f);
  }();
  return fn;
}

// 3-D map of a bf16 [rows, heads, D] tensor with 64 x 1 x 64 boxes (a box at x = 64 of a
// D = 64 tensor lies wholly outside it and reads zeros).
bool encode_rows_tmap(void* tmap, const void* base, int rows, int heads, int D) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)heads, (cuuint64_t)rows};
  const cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)heads * D * 2};
  const cuuint32_t box[3] = {64, 1, 64};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(static_cast<CUtensorMap*>(tmap), CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
            const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_state_tmap(void* tmap, const float* base, int rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)kDk, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)kDk * 4};
  const cuuint32_t box[2] = {32, 32};
  const cuuint32_t estr[2] = {1, 1};
  return fn(static_cast<CUtensorMap*>(tmap), CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2,
            const_cast<float*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_2d_tmap(void* tmap, const void* base, bool bf16, int cols, int rows, int box_cols,
                    int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t esz = bf16 ? 2 : 4;
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)cols * esz};
  const cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(static_cast<CUtensorMap*>(tmap),
            bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2,
            const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace gdn

namespace {

bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

int check_desc_impl(const gdn_desc* d) {
  if (!d) return GDN_ERR_NULL_ARG;
  if (d->T < 0 || d->N < 1 || d->H < 1 || d->Hv < 1 || d->nt_max < 0) return GDN_ERR_BAD_SHAPE;
  if (d->Hv % d->H != 0) return GDN_ERR_BAD_SHAPE;
  if (d->dk != d->dv || (d->dk != 128 && d->dk != 64) || d->chunk_size != kChunk)
    return GDN_ERR_UNSUPPORTED;
  const bool dt_ok = (d->qkv_dtype == GDN_F32 || d->qkv_dtype == GDN_BF16) &&
                     (d->out_dtype == GDN_F32 || d->out_dtype == GDN_BF16);
  if (!dt_ok) return GDN_ERR_UNSUPPORTED;
  if (d->flags & ~(uint32_t)(GDN_FLAG_QK_L2NORM | GDN_FLAG_BUILD_CHUNK_INDICES |
                             GDN_FLAG_CHANNEL_GATES | GDN_FLAG_WORKSPACE_GUARDS))
    return GDN_ERR_UNSUPPORTED;
  // Index arithmetic stays within 64-bit sizes and 32-bit grid limits.
  if ((int64_t)d->T * d->Hv * kDv >= ((int64_t)1 << 40)) return GDN_ERR_BAD_SHAPE;
  if (d->N > 65535 * 16 || d->Hv > 65535 || d->H > 65535) return GDN_ERR_BAD_SHAPE;
  return GDN_OK;
}

int nt_max_of(const gdn_desc* d) {
  return d->nt_max > 0 ? d->nt_max : gdn_nt_max(d->T, d->N, kChunk);
}

bool channel_gates(const gdn_desc* d) { return (d->flags & GDN_FLAG_CHANNEL_GATES) != 0; }

// The tensor-core path serves bf16 inputs (a head of 64 zero-padded to 128; per-channel
// gates through their own intra kernel and the scan's per-channel mode); fp32 inputs
// take the fp32 SIMT path.
bool uses_tc_path(const gdn_desc* d) { return d->qkv_dtype == GDN_BF16; }

// The token-serial and front-end kernels are built for dk = dv = 128 and scalar gates.
bool serial_shape_ok(const gdn_desc* d) { return d->dk == kDk && !channel_gates(d); }

// Guard gap after every workspace region with GDN_FLAG_WORKSPACE_GUARDS.
constexpr size_t kGuardBytes = 4096;
size_t guard_of(const gdn_desc* d) {
  return (d->flags & GDN_FLAG_WORKSPACE_GUARDS) ? kGuardBytes : 0;
}

WsLayout layout_of(const gdn_desc* d) {
  return ws_layout(d->T, d->N, d->H, d->Hv, nt_max_of(d), uses_tc_path(d),
                   (d->flags & GDN_FLAG_QK_L2NORM) != 0, d->dk, channel_gates(d), guard_of(d));
}

// Workspace of the backward pass: the forward's layout (the tensor-core path's for bf16
// inputs, the SIMT path's for fp32), then the chunk-start states and v_new the
// recompute keeps, then the backward intermediates (per slot = chunk slot * Hv + value
// head).
struct BwdLayout {
  WsLayout fwd;
  size_t hs, vn, dvn, dhs, dos, dw, ys, sdot, ttdw, dqp, dkp, total;
};

BwdLayout bwd_layout_of(const gdn_desc* d) {
  BwdLayout B{};
  B.fwd = ws_layout(d->T, d->N, d->H, d->Hv, nt_max_of(d), uses_tc_path(d), false, d->dk,
                    false, guard_of(d));
  size_t o = B.fwd.total;
  auto take = [&](size_t bytes) {
    size_t at = o;
    o = align_up(o + bytes, 256) + guard_of(d);
    return at;
  };
  const size_t slots = (size_t)nt_max_of(d) * d->Hv, D = (size_t)d->dk;
  const size_t mat = sizeof(float) * slots * kChunk * D, st = sizeof(float) * slots * D * D;
  B.hs = take(st);
  B.vn = take(mat);
  B.dvn = take(mat);
  B.dhs = take(st);
  B.dos = take(mat);
  B.dw = take(mat);
  B.ys = take(mat);
  B.sdot = take(sizeof(float) * slots);
  B.ttdw = take(mat);
  B.dqp = take(mat);
  B.dkp = take(mat);
  B.total = o;
  return B;
}

// The backward pass takes scalar gates and no q/k L2 norm.
int check_bwd_desc_impl(const gdn_desc* d) {
  const int rc = check_desc_impl(d);
  if (rc != GDN_OK) return rc;
  if (d->flags & (GDN_FLAG_CHANNEL_GATES | GDN_FLAG_QK_L2NORM)) return GDN_ERR_UNSUPPORTED;
  return GDN_OK;
}

}  // namespace

extern "C" {

int gdn_check_desc(const gdn_desc* desc) { return check_desc_impl(desc); }

int32_t gdn_nt_max(int32_t T, int32_t N, int32_t chunk_size) {
  if (T < 0 || N < 1 || chunk_size < 1) return -1;
  return (int32_t)(((int64_t)T + chunk_size - 1) / chunk_size + N - 1);
}

size_t gdn_workspace_size(const gdn_desc* desc) {
  if (check_desc_impl(desc) != GDN_OK) return 0;
  return layout_of(desc).total;
}

int gdn_build_chunk_indices(const int32_t* cu_seqlens, int32_t N, int32_t T, int32_t nt_max,
                            int32_t* chunk_indices, int32_t* chunk_offsets, int32_t* status,
                            cudaStream_t stream) {
  if (!chunk_offsets) return GDN_ERR_NULL_ARG;
  if (N < 1 || T < 0 || nt_max < 0) return GDN_ERR_BAD_SHAPE;
  if (!cu_seqlens && N != 1) return GDN_ERR_BAD_SHAPE;
  if (!aligned(cu_seqlens, 4) || !aligned(chunk_indices, 8) || !aligned(chunk_offsets, 4) ||
      !aligned(status, 4))
    return GDN_ERR_MISALIGNED;
  launch_chunk_table(cu_seqlens, N, T, nt_max, reinterpret_cast<int2*>(chunk_indices),
                     chunk_offsets, nullptr, status, stream);
  return cudaPeekAtLastError() == cudaSuccess ? GDN_OK : GDN_ERR_LAUNCH_FAILED;
}

int gdn_chunk_fwd(const gdn_desc* desc, const void* q, const void* k, const void* v,
                  const float* g, const float* beta, float scale, const float* initial_state,
                  const int32_t* cu_seqlens, int32_t* chunk_indices, void* out,
                  float* final_state, cudaStream_t stream) {
  int rc = check_desc_impl(desc);
  if (rc != GDN_OK) return rc;
  const gdn_desc& d = *desc;
  if (!q || !k || !v || !g || !beta || !out || !d.workspace) return GDN_ERR_NULL_ARG;
  if (!cu_seqlens && d.N != 1) return GDN_ERR_BAD_SHAPE;
  const bool build_into_caller = chunk_indices && (d.flags & GDN_FLAG_BUILD_CHUNK_INDICES);
  const void* ptrs16[] = {q, k, v, g, beta, out, initial_state, final_state};
  for (const void* p : ptrs16)
    if (!aligned(p, 16)) return GDN_ERR_MISALIGNED;
  if (!aligned(cu_seqlens, 4) || !aligned(chunk_indices, 8)) return GDN_ERR_MISALIGNED;
  if (!aligned(d.workspace, 256)) return GDN_ERR_MISALIGNED;
  const WsLayout L = layout_of(&d);
  if (d.workspace_bytes < L.total) return GDN_ERR_WORKSPACE_TOO_SMALL;

  char* ws = static_cast<char*>(d.workspace);
  const int nt_max = nt_max_of(&d);
  const bool bf16 = d.qkv_dtype == GDN_BF16;
  const bool l2 = (d.flags & GDN_FLAG_QK_L2NORM) != 0;
  if (!(scale > 0.f)) scale = 1.0f / sqrtf((float)d.dk);  // also NaN
  const float eps = d.l2norm_eps > 0.f ? d.l2norm_eps : 1e-6f;

  Params p{};
  p.T = d.T; p.N = d.N; p.H = d.H; p.Hv = d.Hv; p.HG = d.Hv / d.H; p.nt_max = nt_max;
  p.D = d.dk;
  p.q = q; p.k = k; p.v = v; p.g = g; p.beta = beta; p.scale = scale;
  p.s0 = initial_state; p.out = out; p.sT = final_state;
  p.status = reinterpret_cast<int32_t*>(ws + L.status);
  p.seq_info = reinterpret_cast<const int2*>(ws + L.seq_info);
  p.chunk_offsets = reinterpret_cast<const int32_t*>(ws + L.chunk_offsets);
  int2* table = chunk_indices ? reinterpret_cast<int2*>(chunk_indices)
                              : reinterpret_cast<int2*>(ws + L.chunk_table);
  p.chunk_table = table;
  p.seq_order = (d.N > 1 && d.N <= kMaxOrderedSeqs)
                    ? reinterpret_cast<const int32_t*>(ws + L.seq_order)
                    : nullptr;
  p.G = L.G ? reinterpret_cast<float*>(ws + L.G) : nullptr;
  p.EF = L.EF ? reinterpret_cast<float*>(ws + L.EF) : nullptr;
  p.w = ws + L.w;
  p.u = reinterpret_cast<float*>(ws + L.u);
  p.M = ws + L.M;
  p.k16 = L.k16 ? ws + L.k16 : nullptr;
  p.qimg = L.qimg ? ws + L.qimg : nullptr;
  p.q16 = L.q16 ? ws + L.q16 : nullptr;
  p.qt = L.qt ? reinterpret_cast<float*>(ws + L.qt) : nullptr;
  p.kt = L.kt ? reinterpret_cast<float*>(ws + L.kt) : nullptr;
  p.gam = L.gam ? reinterpret_cast<float*>(ws + L.gam) : nullptr;
  p.qrn = l2 ? reinterpret_cast<float*>(ws + L.qrn) : nullptr;
  p.krn = l2 ? reinterpret_cast<float*>(ws + L.krn) : nullptr;
  p.m_f16 = 1;  // the scan takes M v_new on fp16 operands
  p.cu = cu_seqlens;
  p.early_one = d.N == 1 && (!chunk_indices || build_into_caller);
  {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && sms > 0)
      p.pf_ahead = (2 * sms + d.H - 1) / d.H;  // two intra CTAs per SM, key head fastest
    // The intra grid's (key head, slot) CTAs fill 2 x SMs places per wave; when the last
    // wave is partial, its slots are split by value-head halves so that it ends sooner.
    if (sms > 0 && p.HG % 2 == 0) {
      const long items = (long)d.H * nt_max, places = 2L * sms, tail = items % places;
      if (items > places && tail > 0) {
        const int ns = (int)((tail + d.H - 1) / d.H);
        if (nt_max + ns <= 65535) p.split_slots = ns;
      }
    }
  }
  p.out_bf16 = d.out_dtype == GDN_BF16;
  p.stall_polls = scan_stall_polls();
  p.dbg_poison = debug_poison();

  cudaEvent_t* ev = d.stage_events;
  if (ev) cudaEventRecord(ev[0], stream);
  if (l2) launch_l2norm(q, k, bf16, d.T, d.H, d.dk, eps, const_cast<float*>(p.qrn),
                        const_cast<float*>(p.krn), stream);
  launch_chunk_table(cu_seqlens, d.N, d.T, nt_max,
                     (!chunk_indices || build_into_caller) ? table : nullptr,
                     const_cast<int32_t*>(p.chunk_offsets), const_cast<int2*>(p.seq_info),
                     p.status, stream, /*zero_status=*/true,  // (no separate memset)
                     const_cast<int32_t*>(p.seq_order));
  if (ev) cudaEventRecord(ev[1], stream);
  const bool tc = uses_tc_path(&d);
  if (nt_max > 0) {
    if (tc) {
      if (!(channel_gates(&d) ? launch_kda_intra(p, stream) : launch_tc_intra(p, stream)))
        return GDN_ERR_LAUNCH_FAILED;
    } else if (!launch_gen_intra(p, d.dk, channel_gates(&d), bf16, stream)) {
      return GDN_ERR_LAUNCH_FAILED;
    }
  }
  if (ev) cudaEventRecord(ev[2], stream);
  if (tc) {
    if (!launch_tc_inter(p, channel_gates(&d), stream)) return GDN_ERR_LAUNCH_FAILED;
  } else if (!launch_gen_inter(p, d.dk, stream)) {
    return GDN_ERR_LAUNCH_FAILED;
  }
  if (ev) cudaEventRecord(ev[3], stream);
  return cudaPeekAtLastError() == cudaSuccess ? GDN_OK : GDN_ERR_LAUNCH_FAILED;
}

size_t gdn_bwd_workspace_size(const gdn_desc* desc) {
  if (check_bwd_desc_impl(desc) != GDN_OK) return 0;
  return bwd_layout_of(desc).total;
}

int gdn_chunk_bwd(const gdn_desc* desc, const void* q, const void* k, const void* v,
                  const float* g, const float* beta, float scale, const float* initial_state,
                  const int32_t* cu_seqlens, int32_t* chunk_indices, const void* d_out,
                  const float* d_final_state, float* dq, float* dk, float* dv, float* dg,
                  float* dbeta, float* d_initial_state, cudaStream_t stream) {
  int rc = check_bwd_desc_impl(desc);
  if (rc != GDN_OK) return rc;
  const gdn_desc& d = *desc;
  if (!q || !k || !v || !g || !beta || !d_out || !dq || !dk || !dv || !dg || !dbeta ||
      !d.workspace)
    return GDN_ERR_NULL_ARG;
  if (!cu_seqlens && d.N != 1) return GDN_ERR_BAD_SHAPE;
  const bool build_into_caller = chunk_indices && (d.flags & GDN_FLAG_BUILD_CHUNK_INDICES);
  const void* ptrs16[] = {q, k, v, g, beta, d_out, initial_state, d_final_state,
                          dq, dk, dv, dg, dbeta, d_initial_state};
  for (const void* p : ptrs16)
    if (!aligned(p, 16)) return GDN_ERR_MISALIGNED;
  if (!aligned(cu_seqlens, 4) || !aligned(chunk_indices, 8)) return GDN_ERR_MISALIGNED;
  if (!aligned(d.workspace, 256)) return GDN_ERR_MISALIGNED;
  const BwdLayout B = bwd_layout_of(&d);
  if (d.workspace_bytes < B.total) return GDN_ERR_WORKSPACE_TOO_SMALL;

  char* ws = static_cast<char*>(d.workspace);
  const WsLayout& L = B.fwd;
  const int nt_max = nt_max_of(&d), D = d.dk;
  const bool bf16 = d.qkv_dtype == GDN_BF16;
  if (!(scale > 0.f)) scale = 1.0f / sqrtf((float)D);  // also NaN
  auto f32 = [&](size_t off) { return reinterpret_cast<float*>(ws + off); };

  // forward recompute: the SIMT intra kernel and the scan, keeping S and v_new per chunk
  Params p{};
  p.T = d.T; p.N = d.N; p.H = d.H; p.Hv = d.Hv; p.HG = d.Hv / d.H; p.nt_max = nt_max;
  p.D = D;
  p.q = q; p.k = k; p.v = v; p.g = g; p.beta = beta; p.scale = scale;
  p.s0 = initial_state; p.out = nullptr; p.sT = nullptr;
  p.status = reinterpret_cast<int32_t*>(ws + L.status);
  p.seq_info = reinterpret_cast<const int2*>(ws + L.seq_info);
  p.chunk_offsets = reinterpret_cast<const int32_t*>(ws + L.chunk_offsets);
  int2* table = chunk_indices ? reinterpret_cast<int2*>(chunk_indices)
                              : reinterpret_cast<int2*>(ws + L.chunk_table);
  p.chunk_table = table;
  p.seq_order = (d.N > 1 && d.N <= kMaxOrderedSeqs)
                    ? reinterpret_cast<const int32_t*>(ws + L.seq_order)
                    : nullptr;
  const bool tc = uses_tc_path(&d);
  p.w = ws + L.w; p.u = f32(L.u); p.M = ws + L.M;
  p.G = L.G ? f32(L.G) : nullptr;
  p.EF = L.EF ? f32(L.EF) : nullptr;
  p.k16 = L.k16 ? ws + L.k16 : nullptr;
  p.q16 = L.q16 ? ws + L.q16 : nullptr;
  p.qt = L.qt ? f32(L.qt) : nullptr;
  p.kt = L.kt ? f32(L.kt) : nullptr;
  p.gam = L.gam ? f32(L.gam) : nullptr;
  p.hs = f32(B.hs); p.vn_out = f32(B.vn);
  p.stall_polls = scan_stall_polls();
  p.dbg_poison = debug_poison();
  cudaEvent_t* ev = d.stage_events;
  if (ev) cudaEventRecord(ev[0], stream);
  launch_chunk_table(cu_seqlens, d.N, d.T, nt_max,
                     (!chunk_indices || build_into_caller) ? table : nullptr,
                     const_cast<int32_t*>(p.chunk_offsets), const_cast<int2*>(p.seq_info),
                     p.status, stream, /*zero_status=*/true,  // (no separate memset)
                     const_cast<int32_t*>(p.seq_order));
  if (tc) {  // the tensor-core forward kernels, storing S and v_new per chunk
    if (nt_max > 0 && !launch_tc_intra(p, stream)) return GDN_ERR_LAUNCH_FAILED;
    if (!launch_tc_inter(p, false, stream)) return GDN_ERR_LAUNCH_FAILED;
  } else {
    if (nt_max > 0 && !launch_gen_intra(p, D, false, bf16, stream)) return GDN_ERR_LAUNCH_FAILED;
    if (!launch_gen_inter(p, D, stream)) return GDN_ERR_LAUNCH_FAILED;
  }
  if (ev) cudaEventRecord(ev[1], stream);

  BwdParams b{};
  b.T = d.T; b.N = d.N; b.H = d.H; b.Hv = d.Hv; b.HG = p.HG; b.nt_max = nt_max;
  b.q = q; b.k = k; b.v = v; b.g = g; b.beta = beta; b.scale = scale;
  b.dout = d_out; b.dout_bf16 = d.out_dtype == GDN_BF16; b.dfin = d_final_state;
  b.dq = dq; b.dk = dk; b.dv = dv; b.dg = dg; b.dbeta = dbeta; b.dh0 = d_initial_state;
  b.status = p.status; b.seq_info = p.seq_info; b.chunk_offsets = p.chunk_offsets;
  b.chunk_table = table;
  if (tc) {
    b.wimg = ws + L.w; b.mimg = ws + L.M; b.G = p.G;
  } else {
    b.wT = f32(L.w); b.kt = p.kt; b.qt = p.qt; b.MT = f32(L.M); b.gam = p.gam;
  }
  b.hs = p.hs; b.vn = p.vn_out;
  b.dvn = f32(B.dvn); b.dhs = f32(B.dhs); b.dos = f32(B.dos); b.dw = f32(B.dw);
  b.ys = f32(B.ys); b.sdot = f32(B.sdot); b.ttdw = f32(B.ttdw);
  b.dqp = f32(B.dqp); b.dkp = f32(B.dkp);
  if (!launch_bwd(b, D, bf16, tc, stream, ev ? ev + 2 : nullptr)) return GDN_ERR_LAUNCH_FAILED;
  return cudaPeekAtLastError() == cudaSuccess ? GDN_OK : GDN_ERR_LAUNCH_FAILED;
}

int gdn_recurrent_fwd(const gdn_desc* desc, const void* q, const void* k, const void* v,
                      const float* g, const float* beta, float scale,
                      const float* initial_state, const int32_t* cu_seqlens, void* out,
                      float* final_state, cudaStream_t stream) {
  int rc = check_desc_impl(desc);
  if (rc != GDN_OK) return rc;
  if (!serial_shape_ok(desc)) return GDN_ERR_UNSUPPORTED;
  const gdn_desc& d = *desc;
  if (!q || !k || !v || !g || !beta || !out) return GDN_ERR_NULL_ARG;
  if (!cu_seqlens && d.N != 1) return GDN_ERR_BAD_SHAPE;
  const void* ptrs16[] = {q, k, v, g, beta, out, initial_state, final_state};
  for (const void* p : ptrs16)
    if (!aligned(p, 16)) return GDN_ERR_MISALIGNED;
  if (!aligned(cu_seqlens, 4) || !aligned(d.workspace, 256)) return GDN_ERR_MISALIGNED;
  RecParams p{};
  p.T = d.T; p.N = d.N; p.H = d.H; p.Hv = d.Hv; p.HG = d.Hv / d.H;
  p.q = q; p.k = k; p.v = v; p.g = g; p.beta = beta;
  p.scale = scale > 0.f ? scale : 1.0f / sqrtf((float)kDk);  // also NaN
  p.eps = d.l2norm_eps > 0.f ? d.l2norm_eps : 1e-6f;
  p.s0 = initial_state; p.out = out; p.sT = final_state; p.cu = cu_seqlens;
  p.status = d.workspace ? static_cast<int32_t*>(d.workspace) : nullptr;
  p.bf16_in = d.qkv_dtype == GDN_BF16;
  p.out_bf16 = d.out_dtype == GDN_BF16;
  p.l2norm = (d.flags & GDN_FLAG_QK_L2NORM) != 0;
  if (p.status && cudaMemsetAsync(p.status, 0, sizeof(int32_t), stream) != cudaSuccess)
    return GDN_ERR_LAUNCH_FAILED;
  if (d.T > 0 && !launch_recurrent(p, stream)) return GDN_ERR_LAUNCH_FAILED;
  return cudaPeekAtLastError() == cudaSuccess ? GDN_OK : GDN_ERR_LAUNCH_FAILED;
}

int gdn_conv_front(const gdn_desc* desc, const void* x, const float* conv_w, int32_t d_conv,
                   const float* conv_state_in, const int32_t* cu_seqlens, void* q, void* k,
                   void* v, float* conv_state_out, float* snapshots, int32_t n_snapshots,
                   cudaStream_t stream) {
  int rc = check_desc_impl(desc);
  if (rc != GDN_OK) return rc;
  if (desc->dk != kDk) return GDN_ERR_UNSUPPORTED;
  const gdn_desc& d = *desc;
  if (!x || !conv_w || !q || !k || !v) return GDN_ERR_NULL_ARG;
  if (d_conv < 1 || d_conv > 8 || n_snapshots < 0) return GDN_ERR_BAD_SHAPE;
  if ((n_snapshots > 0) != (snapshots != nullptr)) return GDN_ERR_BAD_SHAPE;
  if (!cu_seqlens && d.N != 1) return GDN_ERR_BAD_SHAPE;
  const void* ptrs16[] = {x, q, k, v};
  for (const void* p : ptrs16)
    if (!aligned(p, 16)) return GDN_ERR_MISALIGNED;
  const void* ptrs4[] = {conv_w, conv_state_in, conv_state_out, snapshots, cu_seqlens};
  for (const void* p : ptrs4)
    if (!aligned(p, 4)) return GDN_ERR_MISALIGNED;
  if (!aligned(d.workspace, 256)) return GDN_ERR_MISALIGNED;
  ConvParams p{};
  p.T = d.T; p.N = d.N; p.H = d.H; p.Hv = d.Hv;
  p.C = 2 * d.H * kDk + d.Hv * kDv;
  p.d = d_conv; p.n_snap = n_snapshots;
  p.x = x; p.w = conv_w; p.s_in = conv_state_in; p.s_out = conv_state_out; p.snaps = snapshots;
  p.q = q; p.k = k; p.v = v; p.cu = cu_seqlens;
  p.status = d.workspace ? static_cast<int32_t*>(d.workspace) : nullptr;
  p.eps = d.l2norm_eps > 0.f ? d.l2norm_eps : 1e-6f;
  p.bf16 = d.qkv_dtype == GDN_BF16;
  p.l2norm = (d.flags & GDN_FLAG_QK_L2NORM) != 0;
  if (p.status && cudaMemsetAsync(p.status, 0, sizeof(int32_t), stream) != cudaSuccess)
    return GDN_ERR_LAUNCH_FAILED;
  if (!launch_conv_front(p, stream)) return GDN_ERR_LAUNCH_FAILED;
  return cudaPeekAtLastError() == cudaSuccess ? GDN_OK : GDN_ERR_LAUNCH_FAILED;
}

int gdn_workspace_regions(const gdn_desc* desc, size_t* begin, size_t* end, int max_regions) {
  const int rc = check_desc_impl(desc);
  if (rc != GDN_OK) return rc;
  if (max_regions < 0 || (max_regions > 0 && (!begin || !end))) return GDN_ERR_NULL_ARG;
  const WsLayout L = layout_of(desc);
  for (int i = 0; i < L.nreg && i < max_regions; ++i) {
    begin[i] = L.rbeg[i];
    end[i] = L.rend[i];
  }
  return L.nreg;
}

int gdn_read_status(const gdn_desc* desc, int32_t* host_status, cudaStream_t stream) {
  int rc = check_desc_impl(desc);
  if (rc != GDN_OK) return rc;
  if (!host_status || !desc->workspace) return GDN_ERR_NULL_ARG;
  const WsLayout L = layout_of(desc);
  const char* ws = static_cast<const char*>(desc->workspace);
  if (cudaMemcpyAsync(host_status, ws + L.status, sizeof(int32_t), cudaMemcpyDeviceToHost,
                      stream) != cudaSuccess)
    return GDN_ERR_LAUNCH_FAILED;
  return GDN_OK;
}

int gdn_debug_build(void) {
#ifdef GDN_DEBUG
  return 1;
#else
  return 0;
#endif
}

void gdn_test_debug_poison(int32_t on) {
  g_debug_poison.store(on ? 1 : 0, std::memory_order_relaxed);
}

void gdn_test_scan_timeout(uint32_t polls) {
  g_scan_stall_polls.store(polls, std::memory_order_relaxed);
}

const char* gdn_status_string(int status) {
  switch (status) {
    case GDN_OK: return "ok";
    case GDN_ERR_NULL_ARG: return "a required pointer is NULL";
    case GDN_ERR_BAD_SHAPE: return "invalid dimensions";
    case GDN_ERR_UNSUPPORTED: return "unsupported head size, chunk size, dtype or flag";
    case GDN_ERR_MISALIGNED: return "misaligned pointer";
    case GDN_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case GDN_ERR_LAUNCH_FAILED: return "CUDA launch or copy failed";
    default: return "unknown status";
  }
}

}  // extern "C"
