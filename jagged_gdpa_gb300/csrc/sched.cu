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
constexpr int kSmemBase = 6144;  // segments whose item prefix is searched in shared memory

__device__ __forceinline__ bool direct_dq(const SchedParams& p, const Seg& s) {
  return p.one_tile && dq_direct_segment(s.lq, s.lkv, p.window);
}
__device__ __forceinline__ bool kv_resident(const SchedParams& p, const Seg& s) {
  return p.one_tile && kv_resident_segment(s.lq, s.lkv, p.window);
}

// Items of segment s in a list of this kind; `stored` tells whether the
// segment's dS tiles fit the scratch (used by the two split query lists).
// Segments whose dQ the key-major pass forms directly have no query items.
__device__ int items_of_segment(const SchedParams& p, int kind, const Seg& s, bool stored) {
  if (kind == kUnitsFwd) return kv_resident(p, s) ? 0 : ceil_div(s.lq, 2 * kTile);
  if (kind == kUnitsFwdKvRes) return kv_resident(p, s) ? ceil_div(ceil_div(s.lq, kTile), kChunkTiles) : 0;
  if (kind == kUnitsKvChunk) return ceil_div(ceil_div(s.lkv, kTile), kChunkTiles);
  if (kind == kUnitsKvDirect) return direct_dq(p, s) ? 1 : 0;
  if (kind == kUnitsKv) return direct_dq(p, s) ? 0 : ceil_div(s.lkv, kTile);
  if (direct_dq(p, s)) return 0;
  if (kind == kUnitsQStored && !stored) return 0;
  if (kind == kUnitsQRecompute && stored) return 0;
  return ceil_div(s.lq, kTile);
}

// dS tiles of segment s in the scratch: H nk span (see ds_span); none for a
// segment whose dQ the key-major pass forms directly.
__device__ long long ds_tiles_of_segment(const SchedParams& p, const Seg& s) {
  if (direct_dq(p, s)) return 0;
  return static_cast<long long>(p.heads) * ceil_div(s.lkv, kTile) * ds_span(ceil_div(s.lq, kTile), p.window);
}

__device__ int cost_of_item(int kind, const Seg& s, int tile, int causal, int window) {
  if (kind == kUnitsFwd) {
    const int t0 = 2 * tile, t1 = 2 * tile + 1;
    int c = kv_span_for_q_tile(t0, s.lkv, causal, window).count + 1;
    if (s.lq > t1 * kTile) c += kv_span_for_q_tile(t1, s.lkv, causal, window).count + 1;
    return c;
  }
  if (kind == kUnitsKv || kind == kUnitsKvDirect) return q_span_for_kv_tile(tile, s.lq, causal, window).count + 1;
  if (kind == kUnitsKvChunk) return min(kChunkTiles, ceil_div(s.lkv, kTile) - tile * kChunkTiles) + 1;
  if (kind == kUnitsFwdKvRes) return min(kChunkTiles, ceil_div(s.lq, kTile) - tile * kChunkTiles) + 1;
  return kv_span_for_q_tile(tile, s.lkv, causal, window).count + 1;  // the query lists
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
  __shared__ int32_t base_sm[kSmemBase];
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

  // ---- items per segment, exclusive prefix sum into base[].  With a stored
  // dS scratch the dS tiles are laid out in segment order (H nk span tiles per
  // segment, span: ds_span); a segment is stored when its tiles end within
  // the caller's capacity, so the stored segments are a prefix of the batch.
  // The key list's CTA writes each segment's first tile (-1: not stored);
  // every CTA recomputes the same prefix for its own decisions.
  const bool split_q = L.kind == kUnitsQStored || L.kind == kUnitsQRecompute;
  const bool ds_prefix = p.ds_base != nullptr && (blockIdx.x == 0 || split_q);
  __shared__ long long warp_tot64[32];
  __shared__ long long carry64;
  if (tid == 0) carry64 = 0;
  __syncthreads();
  for (int c0 = 0; c0 < p.batch; c0 += kSchedThreads) {
    const int b = c0 + tid;
    const Seg sg = b < p.batch ? load_seg(p.q_off, p.kv_off, b) : Seg{0, 0, 0, 0};
    bool stored = false;
    if (ds_prefix) {
      const long long need = b < p.batch ? ds_tiles_of_segment(p, sg) : 0;
      const long long incl64 = carry64 + block_inclusive_scan64(need, warp_tot64);
      stored = incl64 <= p.ds_capacity;
      if (blockIdx.x == 0 && b < p.batch) p.ds_base[b] = (stored && !direct_dq(p, sg)) ? incl64 - need : -1;
      __syncthreads();
      if (tid == kSchedThreads - 1) carry64 = incl64;
      __syncthreads();
    }
    const int v = b < p.batch ? items_of_segment(p, L.kind, sg, stored) : 0;
    const int incl = block_inclusive_scan(v, warp_tot);
    if (b < p.batch) base[b] = carry + incl - v;
    __syncthreads();
    if (tid == kSchedThreads - 1) carry += incl;
    __syncthreads();
  }
  if (ds_prefix && blockIdx.x == 0 && tid == 0) p.ds_base[p.batch] = carry64;
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

  // ---- counting sort of items by decreasing cost.  Each item finds its
  // segment by a binary search over the prefix; the prefix is copied to
  // shared memory first when it fits (each search step is then a shared
  // load instead of a dependent global one).
  const int32_t* sbase = base;
  if (p.batch + 1 <= kSmemBase) {
    for (int b = tid; b <= p.batch; b += kSchedThreads) base_sm[b] = base[b];
    __syncthreads();
    sbase = base_sm;
  }
  auto locate = [&](int it, int& b, int& tile) {
    int lo = 0, hi = p.batch - 1;  // largest b with base[b] <= it
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (sbase[mid] <= it) lo = mid;
      else hi = mid - 1;
    }
    b = lo;
    tile = it - sbase[lo];
  };
  // Items of equal cost are counted and placed with one shared-memory atomic
  // per group of equal buckets in a warp (many units often share one cost,
  // and one atomic per item would serialise on that bucket).  Every lane of a
  // warp walks the same rounds so that the warp-wide matches are complete.
  const int lane = tid & 31;
  auto bucket_of = [&](int it, int& b, int& tile, int& cost) -> int {
    if (it >= n_items) return -1;
    locate(it, b, tile);
    cost = cost_of_item(L.kind, load_seg(p.q_off, p.kv_off, b), tile, p.causal, p.window);
    return kCostBuckets - 1 - min(cost, kCostBuckets - 1);
  };
  for (int c = 0; c < n_items; c += kSchedThreads) {
    int b = 0, tile = 0, cost = 0;
    const int bk = bucket_of(c + tid, b, tile, cost);
    const unsigned grp = __match_any_sync(0xffffffffu, bk);
    if (bk >= 0 && lane == __ffs(grp) - 1) atomicAdd(&hist[bk], __popc(grp));
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
  for (int c = 0; c < n_items; c += kSchedThreads) {
    int b = 0, tile = 0, cost = 0;
    const int bk = bucket_of(c + tid, b, tile, cost);
    const unsigned grp = __match_any_sync(0xffffffffu, bk);
    const int leader = __ffs(grp) - 1;
    int first = 0;
    if (bk >= 0 && lane == leader) first = atomicAdd(&hist[bk], __popc(grp));
    first = __shfl_sync(0xffffffffu, first, leader);
    if (bk < 0) continue;
    const int pos = first + __popc(grp & ((1u << lane) - 1u));
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
