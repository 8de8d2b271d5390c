// Software tile scheduler: validates the offsets and builds, for each kind of
// work unit, a list ordered by decreasing cost (longest-processing-time
// first).  The persistent kernels then walk this list in a serpentine order
// over their CTAs, so short and long segments keep every SM busy -- the
// software-level tile scheduling that took the GDPA kernel from a 6x load
// imbalance to near balance ("Meta redesigns AI training infrastructure ...",
// aiuniverse.news, section "Custom Kernels and 5D Parallelism for
// Trillion-Parameter Scale").
//
// One CTA of 1024 threads per list.  Cost is the number of 128x128 tile
// products a unit performs plus one per output tile (its load/store work);
// the counting sort uses kCostBuckets buckets (costs beyond are clamped).
#include "common.cuh"
#include "ptx.cuh"

namespace jg {

namespace {

constexpr int kSchedThreads = 1024;

__device__ int items_of_segment(int kind, const Seg& s) {
  if (kind == kUnitsFwd) return ceil_div(s.lq, 2 * kTile);
  if (kind == kUnitsKv) return ceil_div(s.lkv, kTile);
  return ceil_div(s.lq, kTile);
}

__device__ int cost_of_item(int kind, const Seg& s, int tile, int causal, int window) {
  if (kind == kUnitsFwd) {
    const int t0 = 2 * tile, t1 = 2 * tile + 1;
    int c = kv_span_for_q_tile(t0, s.lkv, causal, window).count + 1;
    if (s.lq > t1 * kTile) c += kv_span_for_q_tile(t1, s.lkv, causal, window).count + 1;
    return c;
  }
  if (kind == kUnitsKv) return q_span_for_kv_tile(tile, s.lq, causal, window).count + 1;
  return kv_span_for_q_tile(tile, s.lkv, causal, window).count + 1;
}

// Inclusive scan of one value per thread over the whole block.
__device__ int block_inclusive_scan(int v, int* warp_tot) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  if (lane == 31) warp_tot[warp] = v;
  __syncthreads();
  if (warp == 0) {
    int w = warp_tot[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += n;
    }
    warp_tot[lane] = w;
  }
  __syncthreads();
  if (warp > 0) v += warp_tot[warp - 1];
  __syncthreads();
  return v;
}

// The same for 64-bit values.
__device__ long long block_inclusive_scan64(long long v, long long* warp_tot) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  if (lane == 31) warp_tot[warp] = v;
  __syncthreads();
  if (warp == 0) {
    long long w = warp_tot[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const long long n = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += n;
    }
    warp_tot[lane] = w;
  }
  __syncthreads();
  if (warp > 0) v += warp_tot[warp - 1];
  __syncthreads();
  return v;
}

}  // namespace

__global__ void __launch_bounds__(kSchedThreads) sched_kernel(const __grid_constant__ SchedParams p) {
  __shared__ int hist[kCostBuckets];
  __shared__ int warp_tot[32];
  __shared__ int bad;
  __shared__ int carry;

  const SchedList& L = p.list[blockIdx.x];
  int32_t* base = p.item_base + static_cast<int64_t>(blockIdx.x) * (p.batch + 1);
  const int tid = threadIdx.x;

  if (tid == 0) {
    bad = 0;
    carry = 0;
  }
  for (int i = tid; i < kCostBuckets; i += kSchedThreads) hist[i] = 0;
  __syncthreads();

  // ---- validate the offsets
  if (tid == 0) {
    if (p.q_off[0] != 0 || p.kv_off[0] != 0 || p.q_off[p.batch] != p.total_q ||
        p.kv_off[p.batch] != p.total_kv)
      bad = 1;
  }
  for (int b = tid; b < p.batch; b += kSchedThreads) {
    if (p.q_off[b + 1] < p.q_off[b] || p.kv_off[b + 1] < p.kv_off[b]) bad = 1;
  }
  __syncthreads();
  if (bad) {
    if (tid == 0) {
      atomicCAS(p.status, kOk, kErrBadOffsets);
      *L.n_units = 0;
    }
    return;
  }

  // ---- stored dS (backward): first scratch tile of each segment, H nk span
  // tiles per segment (span: ds_span), checked against the caller's capacity
  if (p.ds_base != nullptr && blockIdx.x == 0) {
    __shared__ long long warp_tot64[32];
    __shared__ long long carry64;
    if (tid == 0) carry64 = 0;
    __syncthreads();
    for (int c0 = 0; c0 < p.batch; c0 += kSchedThreads) {
      const int b = c0 + tid;
      long long v = 0;
      if (b < p.batch) {
        const Seg sg = load_seg(p.q_off, p.kv_off, b);
        v = static_cast<long long>(p.heads) * ceil_div(sg.lkv, kTile) * ds_span(ceil_div(sg.lq, kTile), p.window);
      }
      const long long incl = block_inclusive_scan64(v, warp_tot64);
      if (b < p.batch) p.ds_base[b] = carry64 + incl - v;
      __syncthreads();
      if (tid == kSchedThreads - 1) carry64 += incl;
      __syncthreads();
    }
    if (tid == 0) {
      p.ds_base[p.batch] = carry64;
      if (carry64 > p.ds_capacity) {  // the scratch is too small for these lengths
        atomicCAS(p.status, kOk, kErrScratchTooSmall);
        *L.n_units = 0;
      }
    }
    __syncthreads();
    if (carry64 > p.ds_capacity) return;
  }

  // ---- items per segment, exclusive prefix sum into base[]
  for (int c0 = 0; c0 < p.batch; c0 += kSchedThreads) {
    const int b = c0 + tid;
    const int v = b < p.batch ? items_of_segment(L.kind, load_seg(p.q_off, p.kv_off, b)) : 0;
    const int incl = block_inclusive_scan(v, warp_tot);
    if (b < p.batch) base[b] = carry + incl - v;
    __syncthreads();
    if (tid == kSchedThreads - 1) carry += incl;
    __syncthreads();
  }
  const int n_items = carry;
  if (tid == 0) base[p.batch] = n_items;
  __syncthreads();
  const long long n_units = static_cast<long long>(n_items) * p.heads;
  if (n_units > L.max_units) {  // the host sizes the list; this cannot happen for valid offsets
    if (tid == 0) {
      atomicCAS(p.status, kOk, kErrBadOffsets);
      *L.n_units = 0;
    }
    return;
  }

  // ---- counting sort of items by decreasing cost
  auto locate = [&](int it, int& b, int& tile) {
    int lo = 0, hi = p.batch - 1;  // largest b with base[b] <= it
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (base[mid] <= it) lo = mid;
      else hi = mid - 1;
    }
    b = lo;
    tile = it - base[lo];
  };
  for (int it = tid; it < n_items; it += kSchedThreads) {
    int b, tile;
    locate(it, b, tile);
    const int cost = cost_of_item(L.kind, load_seg(p.q_off, p.kv_off, b), tile, p.causal, p.window);
    atomicAdd(&hist[kCostBuckets - 1 - min(cost, kCostBuckets - 1)], 1);
  }
  __syncthreads();
  {
    constexpr int kPer = kCostBuckets / kSchedThreads;
    int v[kPer];
    int sum = 0;
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      v[i] = hist[tid * kPer + i];
      sum += v[i];
    }
    const int incl = block_inclusive_scan(sum, warp_tot);
    int run = incl - sum;
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      hist[tid * kPer + i] = run;
      run += v[i];
    }
  }
  __syncthreads();
  for (int it = tid; it < n_items; it += kSchedThreads) {
    int b, tile;
    locate(it, b, tile);
    const int cost = cost_of_item(L.kind, load_seg(p.q_off, p.kv_off, b), tile, p.causal, p.window);
    const int pos = atomicAdd(&hist[kCostBuckets - 1 - min(cost, kCostBuckets - 1)], 1);
    for (int h = 0; h < p.heads; ++h)
      L.units[static_cast<int64_t>(pos) * p.heads + h] = make_int4(b, h, tile, cost);
  }
  if (tid == 0) *L.n_units = static_cast<int>(n_units);
}

}  // namespace jg

namespace jg {
cudaError_t launch_sched(const SchedParams& p, cudaStream_t stream) {
  sched_kernel<<<p.n_lists, kSchedThreads, 0, stream>>>(p);
  return cudaGetLastError();
}
}  // namespace jg
