// gdn_chunk_fwd_noalloc: the forward pass for callers that cannot allocate
// device memory.
//
// Some callers of this library may not call cudaMalloc (or any allocator)
// at the point where they run the layer: for example a host framework that
// hands out all device memory from its own pre-planned arena and forbids
// other allocations, or a latency-critical serving loop where an allocation
// (which can synchronize the device) is not acceptable. gdn_chunk_fwd needs a
// caller-provided workspace; this entry point instead uses a scratch array
// that lives in the library itself, as a file-scope __device__ array, so the
// caller only passes inputs and outputs.
//
// The array is a fixed GDN_NOALLOC_SCRATCH_BYTES on every GPU that loads the
// library, held until the process exits. All calls share it: two calls that
// may run at the same time on the GPU (different streams, or different host
// threads) race on it and must be serialized by the caller. Nothing in it
// needs to start at zero except the status word, which every call clears; the
// status word of the last call stays readable with gdn_noalloc_read_status.
#include "gdn_common.cuh"

namespace {

constexpr size_t kScratchBytes = (size_t)GDN_NOALLOC_SCRATCH_BYTES;

// Device storage of the scratch. In host code this name is only a stand-in
// for the symbol: its device address comes from cudaGetSymbolAddress below.
__device__ __align__(256) unsigned char gdn_noalloc_scratch[kScratchBytes];

// Device address of the scratch on the current device, looked up on every call with
// that device current (no allocation; after the first lookup on a device, which may
// load the library's device code, it is a table lookup). Not cached, so that a device
// reset, which reloads the module, never leaves a stale address. nullptr on failure.
void* scratch_address() {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, gdn_noalloc_scratch) != cudaSuccess) return nullptr;
  return p;
}

}  // namespace

extern "C" int gdn_chunk_fwd_noalloc(const gdn_desc* desc, const void* q, const void* k,
                                     const void* v, const float* g, const float* beta,
                                     float scale, const float* initial_state,
                                     const int32_t* cu_seqlens, int32_t* chunk_indices,
                                     void* out, float* final_state, cudaStream_t stream) {
  const int rc = gdn_check_desc(desc);
  if (rc != GDN_OK) return rc;
  if (gdn_workspace_size(desc) > kScratchBytes) return GDN_ERR_WORKSPACE_TOO_SMALL;
  void* base = scratch_address();
  if (!base) return GDN_ERR_LAUNCH_FAILED;
  gdn_desc d = *desc;
  d.workspace = base;
  d.workspace_bytes = kScratchBytes;
  return gdn_chunk_fwd(&d, q, k, v, g, beta, scale, initial_state, cu_seqlens, chunk_indices,
                       out, final_state, stream);
}

extern "C" int gdn_noalloc_read_status(int32_t* host_status, cudaStream_t stream) {
  if (!host_status) return GDN_ERR_NULL_ARG;
  const char* base = static_cast<const char*>(scratch_address());
  if (!base) return GDN_ERR_LAUNCH_FAILED;
  // the status word sits at the same offset in every workspace layout
  const size_t off = gdn::ws_layout(0, 1, 1, 1, 0, true, false).status;
  if (cudaMemcpyAsync(host_status, base + off, sizeof(int32_t), cudaMemcpyDeviceToHost,
                      stream) != cudaSuccess)
    return GDN_ERR_LAUNCH_FAILED;
  return GDN_OK;
}
