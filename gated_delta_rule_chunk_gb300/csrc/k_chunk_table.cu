// K1: device-side chunk-index builder.
//
// FLA RFC "Graph capture support for prefill and training", section "Core
// design": chunk-count-sized grids are launched at the static bound NT_max and
// the (sequence id, chunk ordinal) table is filled on the device by a
// searchsorted over the per-sequence chunk counts, with a sentinel in unused
// slots, so no host synchronization is needed.
//
// One CTA of 1024 threads: (0) in a forward or backward call, clear the call's status
// word (in place of a separate memset), (1) sanitize the boundaries: each cu_seqlens entry is
// clamped to [0, T] and raised to the largest entry before it (a prefix maximum), so
// sequence n is [max(c_0..c_n), max(c_0..c_n+1)) -- never overlapping another, empty
// where the input decreases -- and count its chunks, (2) exclusive-scan the counts
// into chunk_offsets, (3) for every slot binary-search the sequence that owns it, (4) for
// up to kMaxOrderedSeqs sequences, rank them by chunk count, longest first.
#include "gdn_common.cuh"

namespace gdn {

__global__ void __launch_bounds__(1024)
chunk_table_kernel(const int32_t* __restrict__ cu, int N, int T, int nt_max,
                   int2* __restrict__ table, int32_t* __restrict__ offsets,
                   int2* __restrict__ seq_info, int32_t* status, bool zero_status,
                   int32_t* __restrict__ seq_order) {
  __shared__ int warp_incl[32];
  __shared__ int cnt_s[kMaxOrderedSeqs];  // chunk counts, for the longest-first order
  __shared__ int warp_max[32];
  __shared__ int carry_s, carry_max_s;
  pdl_release();  // the intra kernel may be scheduled now; it waits for this grid's writes
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  if (tid == 0) {
    carry_s = 0;
    carry_max_s = 0;
    if (zero_status && status) *status = 0;  // the call's status word starts clean
  }
  __syncthreads();
  int bad = 0;
  for (int base = 0; base < N; base += 1024) {
    const int n = base + tid;
    // clamped boundaries, then the inclusive prefix maximum of the starts
    const int a = (n < N && cu) ? cu[n] : 0;
    const int b = n < N ? (cu ? cu[n + 1] : T) : 0;
    int pm = min(max(a, 0), T);
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, pm, o);
      if (lane >= o) pm = max(pm, y);
    }
    if (lane == 31) warp_max[wid] = pm;
    __syncthreads();
    if (wid == 0) {
      int wm = warp_max[lane];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, wm, o);
        if (lane >= o) wm = max(wm, y);
      }
      warp_max[lane] = wm;
    }
    __syncthreads();
    pm = max(max(pm, carry_max_s), wid ? warp_max[wid - 1] : 0);
    int cnt = 0;
    if (n < N) {
      const int s = pm;                          // max(c_0 .. c_n)
      const int e = max(min(max(b, 0), T), s);   // max(c_0 .. c_n+1)
      bad |= (a != s) | (b != e);
      const int len = e - s;
      cnt = (len + kChunk - 1) / kChunk;
      if (seq_info) seq_info[n] = make_int2(s, len);
      if (n < kMaxOrderedSeqs) cnt_s[n] = cnt;
    }
    __syncthreads();
    if (tid == 1023) carry_max_s = pm;
    int x = cnt;  // inclusive warp scan
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) warp_incl[wid] = x;
    __syncthreads();
    if (wid == 0) {
      int ws = warp_incl[lane];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, ws, o);
        if (lane >= o) ws += y;
      }
      warp_incl[lane] = ws;
    }
    __syncthreads();
    const int excl = carry_s + (wid ? warp_incl[wid - 1] : 0) + x - cnt;
    if (n < N && dbg_ok(n <= N, status)) offsets[n] = excl;
    __syncthreads();
    if (tid == 1023) carry_s = excl + cnt;
    __syncthreads();
  }
  const int total = carry_s;
  if (tid == 0) {
    offsets[N] = total;
    if (total > nt_max) set_status(status, GDN_DEV_CHUNK_OVERFLOW);
  }
  if (bad) set_status(status, GDN_DEV_BAD_CU_SEQLENS);
  __syncthreads();  // offsets[] (global) and cnt_s visible to the whole block
  if (seq_order && N <= kMaxOrderedSeqs && tid < N) {
    // (4) the sequences by chunk count, longest first (ties by index): the scan's CTAs of
    // long sequences start first, so that the short ones fill the SMs behind them
    const int mine = cnt_s[tid];
    int rank = 0;
    for (int m = 0; m < N; ++m) {
      const int o = cnt_s[m];
      rank += (o > mine) || (o == mine && m < tid);
    }
    if (dbg_ok(rank < N, status)) seq_order[rank] = tid;
  }
  if (!table) return;
  for (int s = tid; s < nt_max; s += 1024) {
    int2 r = make_int2(-1, -1);
    if (s < total) {
      // offsets[lo] <= s < offsets[hi]; offsets[0] = 0 and offsets[N] = total.
      int lo = 0, hi = N;
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (offsets[mid] <= s) lo = mid; else hi = mid;
      }
      r = make_int2(lo, s - offsets[lo]);
    }
    if (dbg_ok(s < nt_max, status)) table[s] = r;
  }
}

void launch_chunk_table(const int32_t* cu, int N, int T, int nt_max, int2* table,
                        int32_t* offsets, int2* seq_info, int32_t* status, cudaStream_t s,
                        bool zero_status, int32_t* seq_order) {
  chunk_table_kernel<<<1, 1024, 0, s>>>(cu, N, T, nt_max, table, offsets, seq_info, status,
                                        zero_status, N <= kMaxOrderedSeqs ? seq_order : nullptr);
}

}  // namespace gdn
