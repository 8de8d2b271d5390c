// Host side of libjgdpa.so: argument validation, workspace layout, TMA tensor
// maps and kernel launches behind the C ABI declared in include/jgdpa.h.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/jgdpa.h"
#include "act.cuh"
#include "common.cuh"
#include "ptx.cuh"

namespace jg {
// Per-head-dimension launchers, one object file per head dimension.
template <int D>
cudaError_t launch_fwd_d(const FwdParams& p, int act, int grid, cudaStream_t stream);
template <int D>
cudaError_t launch_fwd_shortq_d(const FwdParams& p, int act, int nq, int grid, cudaStream_t stream);
template <int D>
cudaError_t launch_fwd_kvres_d(const FwdParams& p, int act, int grid, cudaStream_t stream);
template <int D>
cudaError_t launch_bwd_pass_d(const BwdParams& p, int act, bool kv_major, int grid, cudaStream_t stream,
                              bool direct);
template <int D>
cudaError_t launch_bwd_shortq_d(const BwdParams& p, int act, int nq, int grid, cudaStream_t stream);
template <int D>
cudaError_t launch_dq_ds_d(const BwdParams& p, int grid, cudaStream_t stream);
template <int D>
cudaError_t launch_softmax_delta_d(const void* out, const void* dout, float* delta, int64_t total_q, int heads,
                                   const int* status, cudaStream_t stream);
cudaError_t launch_dbias_reduce(const unsigned long long* part, float* dbias, int n_parts, int n,
                                cudaStream_t stream);
cudaError_t launch_dq_shared_reduce(const float* part, void* dq, int batch, int64_t n, const int* status,
                                    cudaStream_t stream);
cudaError_t launch_dq_fused_reduce(const float* part, float* tmp, void* dq, const int32_t* item_base, int batch,
                                   int heads, int rows, int d, const int* status, cudaStream_t stream);
size_t dq_fused_tmp_floats(int heads, int rows, int d);
cudaError_t launch_sched(const SchedParams& p, cudaStream_t stream);

cudaError_t launch_fwd(const FwdParams& p, int head_dim, int act, int grid, cudaStream_t stream) {
  if (head_dim == 128) return launch_fwd_d<128>(p, act, grid, stream);
  if (head_dim == 64) return launch_fwd_d<64>(p, act, grid, stream);
  if (head_dim == 32) return launch_fwd_d<32>(p, act, grid, stream);
  return cudaErrorInvalidValue;
}
cudaError_t launch_fwd_shortq(const FwdParams& p, int head_dim, int act, int nq, int grid, cudaStream_t stream) {
  if (head_dim == 128) return launch_fwd_shortq_d<128>(p, act, nq, grid, stream);
  if (head_dim == 64) return launch_fwd_shortq_d<64>(p, act, nq, grid, stream);
  if (head_dim == 32) return launch_fwd_shortq_d<32>(p, act, nq, grid, stream);
  return cudaErrorInvalidValue;
}
// direct: the key-major pass over the units of the direct-dQ segments
cudaError_t launch_bwd_pass(const BwdParams& p, int head_dim, int act, bool kv_major, int grid,
                            cudaStream_t stream, bool direct = false) {
  if (head_dim == 128) return launch_bwd_pass_d<128>(p, act, kv_major, grid, stream, direct);
  if (head_dim == 64) return launch_bwd_pass_d<64>(p, act, kv_major, grid, stream, direct);
  if (head_dim == 32) return launch_bwd_pass_d<32>(p, act, kv_major, grid, stream, direct);
  return cudaErrorInvalidValue;
}
cudaError_t launch_bwd_shortq(const BwdParams& p, int head_dim, int act, int nq, int grid, cudaStream_t stream) {
  if (head_dim == 128) return launch_bwd_shortq_d<128>(p, act, nq, grid, stream);
  if (head_dim == 64) return launch_bwd_shortq_d<64>(p, act, nq, grid, stream);
  if (head_dim == 32) return launch_bwd_shortq_d<32>(p, act, nq, grid, stream);
  return cudaErrorInvalidValue;
}
cudaError_t launch_fwd_kvres(const FwdParams& p, int head_dim, int act, int grid, cudaStream_t stream) {
  if (head_dim == 128) return launch_fwd_kvres_d<128>(p, act, grid, stream);
  if (head_dim == 64) return launch_fwd_kvres_d<64>(p, act, grid, stream);
  if (head_dim == 32) return launch_fwd_kvres_d<32>(p, act, grid, stream);
  return cudaErrorInvalidValue;
}
cudaError_t launch_dq_ds(const BwdParams& p, int head_dim, int grid, cudaStream_t stream) {
  if (head_dim == 128) return launch_dq_ds_d<128>(p, grid, stream);
  if (head_dim == 64) return launch_dq_ds_d<64>(p, grid, stream);
  if (head_dim == 32) return launch_dq_ds_d<32>(p, grid, stream);
  return cudaErrorInvalidValue;
}
cudaError_t launch_softmax_delta(const void* out, const void* dout, float* delta, int64_t total_q, int heads,
                                 int head_dim, const int* status, cudaStream_t stream) {
  if (head_dim == 128) return launch_softmax_delta_d<128>(out, dout, delta, total_q, heads, status, stream);
  if (head_dim == 64) return launch_softmax_delta_d<64>(out, dout, delta, total_q, heads, status, stream);
  return launch_softmax_delta_d<32>(out, dout, delta, total_q, heads, status, stream);
}
}  // namespace jg

namespace {

using jg::kTile;

constexpr size_t kAlign = 256;
constexpr int kShortQMax = 64;  // largest shared query block the short-query kernels take
size_t up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

// Limit of one internal device wait for the kernels launched from now on
// (jgdpa_set_wait_limit_ns; 0 = the default).
std::atomic<unsigned long long> g_wait_limit_ns{0};
unsigned long long wait_limit_ns() {
  const unsigned long long v = g_wait_limit_ns.load(std::memory_order_relaxed);
  return v ? v : jg::kWaitLimitNs;
}

// ----------------------------------------------------------- device facts
int sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  static int cache[128] = {0};
  if (dev < 0 || dev >= 128) return 0;
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    cache[dev] = n;
  }
  return cache[dev];
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link
// dependency on libcuda).
using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                              const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                              CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeFn encode_fn() {
  static std::once_flag once;
  static EncodeFn fn = nullptr;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeFn>(f);
  });
  return fn;
}

// 3-D map over a packed [rows][heads][d] bf16 tensor; box = box_rows (128 by
// default) rows x 1 head x min(d, 64) columns, swizzled to match the MMA
// operand layout.  The last kMapCache encodings are kept (a map holds only
// the address, extents, strides and box, so an entry stays valid for any
// tensor of that address and shape), so that repeated calls with the same
// tensors skip the driver's encode.
constexpr int kMapCache = 64;
struct MapEntry {
  const void* ptr;
  int64_t rows;
  int heads, d, box_rows;
  bool valid;
  CUtensorMap map;
};
std::mutex g_map_mu;
MapEntry g_maps[kMapCache];
int g_map_next = 0;

bool encode_map(CUtensorMap* m, const void* ptr, int64_t rows, int heads, int d, int box_rows);

bool make_map(CUtensorMap* m, const void* ptr, int64_t rows, int heads, int d, int box_rows = kTile) {
  {
    std::lock_guard<std::mutex> lock(g_map_mu);
    for (const MapEntry& e : g_maps)
      if (e.valid && e.ptr == ptr && e.rows == rows && e.heads == heads && e.d == d && e.box_rows == box_rows) {
        *m = e.map;
        return true;
      }
  }
  if (!encode_map(m, ptr, rows, heads, d, box_rows)) return false;
  std::lock_guard<std::mutex> lock(g_map_mu);
  MapEntry& e = g_maps[g_map_next];
  g_map_next = (g_map_next + 1) % kMapCache;
  e = MapEntry{ptr, rows, heads, d, box_rows, true, *m};
  return true;
}

bool encode_map(CUtensorMap* m, const void* ptr, int64_t rows, int heads, int d, int box_rows) {
  std::memset(m, 0, sizeof(*m));
  EncodeFn enc = encode_fn();
  if (!enc || rows <= 0) return false;
  const int box_cols = d < 64 ? d : 64;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(heads), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2, static_cast<cuuint64_t>(heads) * d * 2};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(box_cols), 1, static_cast<cuuint32_t>(box_rows)};
  cuuint32_t es[3] = {1, 1, 1};
  const CUtensorMapSwizzle sw = box_cols * 2 == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D view of the stored-dS scratch: rows of 128 bf16 (one tile row), boxes
// of 64 columns x 128 rows with the 128-byte swizzle (one column block of a
// tile, the shared-memory layout of the kernels' X tiles).
bool make_ds_map(CUtensorMap* m, void* ptr, int64_t tiles) {
  std::memset(m, 0, sizeof(*m));
  EncodeFn enc = encode_fn();
  if (!enc || tiles <= 0) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(kTile), static_cast<cuuint64_t>(tiles) * kTile};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(kTile) * 2};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(kTile / 2), static_cast<cuuint32_t>(kTile)};
  cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, ptr, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// ------------------------------------------------------------- workspace
struct Layout {
  size_t header = 0;      // status word + unit counters
  size_t item_base = 0;   // scheduler scratch, 2 lists x (batch + 1)
  size_t units0 = 0;      // fwd units, or dkdv units
  size_t units1 = 0;      // dq units (bwd): all, or those of the segments with stored dS; fwd: key/value-resident units
  size_t units2 = 0;      // bwd with a dS scratch: dq units of the segments recomputed
  size_t units3 = 0;      // bwd: dkdv units of the segments whose dQ that pass forms directly
  size_t delta = 0;       // softmax bwd: [H][total_q]
  size_t dbias = 0;       // bwd with dbias: [grid][H][T] 64-bit fixed-point partial sums
  size_t ds_base = 0;     // bwd: first stored-dS tile per segment, int64 [batch + 1]
  size_t q_off = 0;       // shared queries: the synthesized query offsets S b, int32 [batch + 1]
  size_t dq_part = 0;     // shared queries, bwd: fp32 dQ of every segment's rows [batch S][H][d]
  size_t dq_fused = 0;    // fused dQ (shared, S <= 128, d <= 64): [key items][H][S][d] fp32 blocks
  size_t dq_fused_tmp = 0;  // its first-stage sums
  bool fused_dq = false;
  size_t total = 0;
  int max0 = 0, max1 = 0;
  int grid = 0;
};

int64_t max_units(int64_t total, int64_t batch, int rows_per_unit, int heads) {
  return (total / rows_per_unit + batch) * heads;
}

// Shared queries with at most one query tile and d <= 64: the key-major pass
// has TMEM room to form each unit's dQ contribution itself, so the backward
// stores no dS and runs no dQ pass (the fused split-dQ).
bool fused_dq_applies(int32_t q_shared, int32_t head_dim) {
  return q_shared > 0 && q_shared <= kTile && head_dim <= 64;
}
// Shared queries of at most kShortQMax rows with GELU / SiLU: the short-query
// backward (keys on the MMA's rows, the queries as N), which also writes one
// fp32 dQ contribution per unit for the same ordered reduction.
bool shortq_bwd_applies(int32_t q_shared, int32_t act) {
  return q_shared > 0 && q_shared <= kShortQMax && act != JGDPA_ACT_SOFTMAX;
}

bool layout_for(int32_t batch, int64_t total_q, int64_t total_kv, int32_t heads, int32_t act, int32_t bias_len,
                bool bwd, Layout* L, int32_t q_shared = 0, int32_t head_dim = 0) {
  const int sms = sm_count();
  if (sms <= 0) return false;
  int64_t m0, m1 = 0;
  if (!bwd) {
    m0 = max_units(total_q, batch, 2 * kTile, heads);
    m1 = max_units(total_q, batch, kTile, heads);  // key/value-resident units (one per query tile at most)
  } else {
    m0 = max_units(total_kv, batch, kTile, heads);
    m1 = max_units(total_q, batch, kTile, heads);
  }
  if (m0 > INT32_MAX / 2 || m1 > INT32_MAX / 2) return false;
  L->max0 = static_cast<int>(m0);
  L->max1 = static_cast<int>(m1);
  L->grid = sms;
  size_t off = 0;
  L->header = off;
  off += up(64 * sizeof(int));
  L->item_base = off;
  off += up(4 * (static_cast<size_t>(batch) + 1) * sizeof(int32_t));
  L->units0 = off;
  off += up(static_cast<size_t>(m0) * sizeof(jg::Unit));
  L->units1 = off;
  off += up(static_cast<size_t>(m1) * sizeof(jg::Unit));
  L->units2 = off;
  if (bwd) off += up(static_cast<size_t>(m1) * sizeof(jg::Unit));
  L->units3 = off;
  if (bwd) off += up(static_cast<size_t>(m0) * sizeof(jg::Unit));
  L->delta = off;
  if (bwd && act == JGDPA_ACT_SOFTMAX) off += up(static_cast<size_t>(heads) * total_q * sizeof(float));
  L->dbias = off;
  if (bwd && bias_len > 0) off += up(static_cast<size_t>(sms) * heads * bias_len * sizeof(unsigned long long));
  L->ds_base = off;
  if (bwd) off += up((static_cast<size_t>(batch) + 1) * sizeof(int64_t));
  L->q_off = off;
  if (q_shared > 0) off += up((static_cast<size_t>(batch) + 1) * sizeof(int32_t));
  L->fused_dq = bwd && (fused_dq_applies(q_shared, head_dim) || shortq_bwd_applies(q_shared, act));
  L->dq_part = off;
  if (q_shared > 0 && bwd && !L->fused_dq)
    off += up(static_cast<size_t>(total_q) * heads * head_dim * sizeof(float));
  L->dq_fused = off;
  L->dq_fused_tmp = off;
  if (L->fused_dq) {
    const size_t items = static_cast<size_t>(m0 / heads);  // key tiles (at least the chunks), all segments
    off += up(items * heads * q_shared * head_dim * sizeof(float));
    L->dq_fused_tmp = off;
    off += up(jg::dq_fused_tmp_floats(heads, q_shared, head_dim) * sizeof(float));
  }
  L->total = off;
  return true;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

jgdpa_status check_common(int32_t batch, int64_t total_q, int64_t total_kv, int32_t heads, int32_t head_dim,
                          int32_t act, float scale, const float* bias_table, int32_t bias_len, int32_t causal,
                          const int32_t* q_offsets, const int32_t* kv_offsets) {
  if (batch < 0 || total_q < 0 || total_kv < 0 || heads < 1) return JGDPA_ERR_INVALID_ARGUMENT;
  if (act < JGDPA_ACT_GELU || act > JGDPA_ACT_SOFTMAX) return JGDPA_ERR_INVALID_ARGUMENT;
  if (causal != 0 && causal != 1) return JGDPA_ERR_INVALID_ARGUMENT;
  if (!std::isfinite(scale)) return JGDPA_ERR_INVALID_ARGUMENT;
  if (bias_len < 0 || (bias_len > 0 && (bias_len % 2 == 0 || bias_table == nullptr)) ||
      (bias_len == 0 && bias_table != nullptr))
    return JGDPA_ERR_INVALID_ARGUMENT;
  if (bias_len > jg::kMaxBiasLen) return JGDPA_ERR_UNSUPPORTED;
  if (head_dim != 32 && head_dim != 64 && head_dim != 128) return JGDPA_ERR_UNSUPPORTED;
  if (total_q > INT32_MAX || total_kv > INT32_MAX || heads > 65535) return JGDPA_ERR_UNSUPPORTED;
  if (batch > 0 && (q_offsets == nullptr || kv_offsets == nullptr)) return JGDPA_ERR_INVALID_ARGUMENT;
  if (batch == 0 && (total_q != 0 || total_kv != 0)) return JGDPA_ERR_INVALID_ARGUMENT;
  if (!aligned(q_offsets, 4) || !aligned(kv_offsets, 4) || !aligned(bias_table, 4)) return JGDPA_ERR_MISALIGNED;
  return JGDPA_OK;
}

#define JG_CUDA(x)                              \
  do {                                          \
    if ((x) != cudaSuccess) return JGDPA_ERR_CUDA; \
  } while (0)

__global__ void fill_f32_kernel(float* p, int64_t n, float v) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i < n) p[i] = v;
}

__global__ void shared_q_offsets_kernel(int32_t* q_off, int32_t batch, int32_t n_shared) {
  const int64_t b = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (b <= batch) q_off[b] = static_cast<int32_t>(b * n_shared);
}

cudaError_t fill_f32(float* p, int64_t n, float v, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  fill_f32_kernel<<<static_cast<unsigned>((n + 255) / 256), 256, 0, s>>>(p, n, v);
  return cudaGetLastError();
}

// Evaluates the kernels' packed activation routines (act2: forward value,
// act2_d: backward derivative) on two elements per thread, from hx = x / 2
// exactly as the kernels form it.
template <int ACT, int PATH>
__device__ void eval_act_pair(const float* x, int64_t i, int64_t n, float* y, float* dy) {
  const float2 hx = make_float2(0.5f * x[i], i + 1 < n ? 0.5f * x[i + 1] : 0.f);
  const float2 a = jg::act2_route<ACT, PATH>(hx);
  float2 d;  // the ex2 route is forward-only: its derivative is the SFU one
  (void)jg::act2_d<ACT, PATH == 1>(hx, d);
  y[i] = a.x;
  if (dy) dy[i] = d.x;
  if (i + 1 < n) {
    y[i + 1] = a.y;
    if (dy) dy[i + 1] = d.y;
  }
}

__global__ void eval_act_kernel(int act, int path, const float* x, int64_t n, float* y, float* dy) {
  const int64_t i = 2 * (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x);
  if (i >= n) return;
  if (act == 0) {
    if (path == 1) eval_act_pair<0, 1>(x, i, n, y, dy);
    else if (path == 2) eval_act_pair<0, 2>(x, i, n, y, dy);
    else eval_act_pair<0, 0>(x, i, n, y, dy);
  } else {
    if (path == 1) eval_act_pair<1, 1>(x, i, n, y, dy);
    else if (path == 2) eval_act_pair<1, 2>(x, i, n, y, dy);
    else eval_act_pair<1, 0>(x, i, n, y, dy);
  }
}

jgdpa_status run_sched(const int32_t* q_off, const int32_t* kv_off, int32_t batch, int32_t heads,
                          int64_t total_q, int64_t total_kv, int32_t causal, int32_t window, uint8_t* ws,
                          const Layout& L, bool bwd, cudaStream_t stream, int64_t ds_capacity = -1,
                          bool kv_chunks = false, bool one_tile = false) {
  jg::SchedParams sp{};
  sp.one_tile = one_tile ? 1 : 0;
  if (ds_capacity >= 0) {
    sp.ds_base = reinterpret_cast<int64_t*>(ws + L.ds_base);
    sp.ds_capacity = ds_capacity;
  }
  sp.q_off = q_off;
  sp.kv_off = kv_off;
  sp.batch = batch;
  sp.heads = heads;
  sp.total_q = total_q;
  sp.total_kv = total_kv;
  sp.causal = causal;
  sp.window = window;
  int* hdr = reinterpret_cast<int*>(ws + L.header);
  sp.status = hdr;
  sp.item_base = reinterpret_cast<int32_t*>(ws + L.item_base);
  // (short-query backward: the key-tile chunks only, no query lists)
  sp.list[0].kind = kv_chunks ? jg::kUnitsKvChunk : (bwd ? jg::kUnitsKv : jg::kUnitsFwd);
  sp.list[0].max_units = L.max0;
  sp.list[0].n_units = hdr + 1;
  sp.list[0].units = reinterpret_cast<jg::Unit*>(ws + L.units0);
  sp.n_lists = kv_chunks ? 1 : (bwd ? (ds_capacity >= 0 ? 3 : 2) : 1);
  if (bwd && !kv_chunks) {
    sp.list[1].kind = ds_capacity >= 0 ? jg::kUnitsQStored : jg::kUnitsQ;
    sp.list[1].max_units = L.max1;
    sp.list[1].n_units = hdr + 2;
    sp.list[1].units = reinterpret_cast<jg::Unit*>(ws + L.units1);
  }
  if (bwd && !kv_chunks && ds_capacity >= 0) {
    sp.list[2].kind = jg::kUnitsQRecompute;
    sp.list[2].max_units = L.max1;
    sp.list[2].n_units = hdr + 3;
    sp.list[2].units = reinterpret_cast<jg::Unit*>(ws + L.units2);
  }
  if (one_tile && !bwd) {  // the key/value-resident forward units
    jg::SchedList& ol = sp.list[sp.n_lists++];
    ol.kind = jg::kUnitsFwdKvRes;
    ol.max_units = L.max1;
    ol.n_units = hdr + 2;
    ol.units = reinterpret_cast<jg::Unit*>(ws + L.units1);
  }
  if (one_tile && bwd) {  // the key-major units of the direct-dQ segments, last list
    jg::SchedList& dl = sp.list[sp.n_lists++];
    dl.kind = jg::kUnitsKvDirect;
    dl.max_units = L.max0;
    dl.n_units = hdr + 4;
    dl.units = reinterpret_cast<jg::Unit*>(ws + L.units3);
  }
  JG_CUDA(jg::launch_sched(sp, stream));
  JG_CUDA(cudaGetLastError());
  return JGDPA_OK;
}

}  // namespace

extern "C" {

size_t jgdpa_workspace_bytes(int32_t batch, int64_t total_q, int64_t total_kv, int32_t heads, int32_t head_dim,
                             jgdpa_act act, int32_t bias_len, int32_t for_backward) {
  if (batch < 0 || total_q < 0 || total_kv < 0 || heads < 1 || bias_len < 0) return 0;
  if (head_dim != 32 && head_dim != 64 && head_dim != 128) return 0;
  Layout L;
  if (!layout_for(batch, total_q, total_kv, heads, act, bias_len, for_backward != 0, &L)) return 0;
  return L.total;
}

}  // extern "C"

namespace {

// q_shared > 0: every segment reads the same q_shared query rows (q is
// [q_shared][H][d]); q_offsets is then ignored and synthesized in the
// workspace as q_shared b, so that O and LSE keep one block of rows per
// segment (total_q = batch q_shared).
jgdpa_status fwd_impl(const void* q, const void* k, const void* v, const int32_t* q_offsets,
                      const int32_t* kv_offsets, int32_t batch, int64_t total_q, int64_t total_kv, int32_t heads,
                      int32_t head_dim, jgdpa_act act, float scale, const float* bias_table, int32_t bias_len,
                      int32_t causal, int32_t window, void* out, float* lse, void* workspace,
                      size_t workspace_bytes, jgdpa_stream_t stream_, int32_t q_shared = 0) {
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  jgdpa_status st = check_common(batch, total_q, total_kv, heads, head_dim, act, scale, bias_table, bias_len,
                                 causal, q_shared > 0 ? kv_offsets : q_offsets, kv_offsets);
  if (st != JGDPA_OK) return st;
  if (window < 0) return JGDPA_ERR_INVALID_ARGUMENT;
  if ((act == JGDPA_ACT_SOFTMAX) != (lse != nullptr)) return JGDPA_ERR_INVALID_ARGUMENT;
  if (total_q > 0 && (q == nullptr || out == nullptr)) return JGDPA_ERR_INVALID_ARGUMENT;
  if (total_kv > 0 && (k == nullptr || v == nullptr)) return JGDPA_ERR_INVALID_ARGUMENT;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16) || !aligned(lse, 4))
    return JGDPA_ERR_MISALIGNED;
  Layout L;
  if (!layout_for(batch, total_q, total_kv, heads, act, bias_len, false, &L, q_shared, head_dim))
    return JGDPA_ERR_CUDA;
  if (workspace == nullptr || workspace_bytes < L.total) return JGDPA_ERR_WORKSPACE_TOO_SMALL;
  if (!aligned(workspace, kAlign)) return JGDPA_ERR_MISALIGNED;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  JG_CUDA(cudaMemsetAsync(ws + L.header, 0, 64 * sizeof(int), stream));
  if (batch == 0 || total_q == 0) return JGDPA_OK;
  if (q_shared > 0) {
    int32_t* qo = reinterpret_cast<int32_t*>(ws + L.q_off);
    shared_q_offsets_kernel<<<static_cast<unsigned>((batch + 1 + 255) / 256), 256, 0, stream>>>(qo, batch, q_shared);
    JG_CUDA(cudaGetLastError());
    q_offsets = qo;
  }
  if (total_kv == 0) {  // no keys anywhere: O = 0, LSE = -inf
    JG_CUDA(cudaMemsetAsync(out, 0, static_cast<size_t>(total_q) * heads * head_dim * 2, stream));
    if (lse) JG_CUDA(fill_f32(lse, total_q * heads, -INFINITY, stream));
    return JGDPA_OK;
  }
  // shared queries of at most 64 rows (GELU / SiLU): keys on the MMA's 128
  // rows and the queries as N, so the activation touches only live elements
  const bool shortq = q_shared > 0 && q_shared <= kShortQMax && act != JGDPA_ACT_SOFTMAX;
  // otherwise the segments whose keys fit one tile and that have two or more
  // query tiles run in the key/value-resident forward
  const bool one_tile = !shortq && window == 0;
  st = run_sched(q_offsets, kv_offsets, batch, heads, total_q, total_kv, causal, window, ws, L, false, stream, -1,
                 false, one_tile);
  if (st != JGDPA_OK) return st;

  jg::FwdParams p{};
  if (!make_map(&p.tm_q, q, q_shared > 0 ? q_shared : total_q, heads, head_dim) ||
      !make_map(&p.tm_k, k, total_kv, heads, head_dim) || !make_map(&p.tm_v, v, total_kv, heads, head_dim))
    return JGDPA_ERR_CUDA;
  p.q_shared = q_shared > 0 ? 1 : 0;
  int* hdr = reinterpret_cast<int*>(ws + L.header);
  p.q_off = q_offsets;
  p.kv_off = kv_offsets;
  p.units = reinterpret_cast<const jg::Unit*>(ws + L.units0);
  p.n_units = hdr + 1;
  p.status = hdr;
  p.bias = bias_table;
  p.out = static_cast<__nv_bfloat16*>(out);
  p.lse = lse;
  p.total_q = total_q;
  p.heads = heads;
  p.bias_len = bias_len;
  p.causal = causal;
  p.window = window;
  p.scale = act == JGDPA_ACT_SOFTMAX ? scale * jg::kLog2e : scale;
  p.wait_limit_ns = wait_limit_ns();
  const int grid = static_cast<int>(std::min<int64_t>(L.grid, std::max(1, L.max0)));
  if (shortq) {
    JG_CUDA(jg::launch_fwd_shortq(p, head_dim, act, q_shared, grid, stream));
  } else {
    // O stores by TMA (32-row boxes) from the staged epilogues
    if (!make_map(&p.tm_o, out, total_q, heads, head_dim, 32)) return JGDPA_ERR_CUDA;
    JG_CUDA(jg::launch_fwd(p, head_dim, act, grid, stream));
    if (one_tile) {
      p.units = reinterpret_cast<const jg::Unit*>(ws + L.units1);
      p.n_units = hdr + 2;
      JG_CUDA(jg::launch_fwd_kvres(p, head_dim, act, grid, stream));
    }
  }
  return JGDPA_OK;
}

}  // namespace

extern "C" {

jgdpa_status jgdpa_fwd(const void* q, const void* k, const void* v, const int32_t* q_offsets,
                       const int32_t* kv_offsets, int32_t batch, int64_t total_q, int64_t total_kv, int32_t heads,
                       int32_t head_dim, jgdpa_act act, float scale, const float* bias_table, int32_t bias_len,
                       int32_t causal, void* out, float* lse, void* workspace, size_t workspace_bytes,
                       jgdpa_stream_t stream) {
  return fwd_impl(q, k, v, q_offsets, kv_offsets, batch, total_q, total_kv, heads, head_dim, act, scale,
                  bias_table, bias_len, causal, 0, out, lse, workspace, workspace_bytes, stream);
}

jgdpa_status jgdpa_fwd_ex(const void* q, const void* k, const void* v, const int32_t* q_offsets,
                          const int32_t* kv_offsets, int32_t batch, int64_t total_q, int64_t total_kv,
                          int32_t heads, int32_t head_dim, jgdpa_act act, float scale, const float* bias_table,
                          int32_t bias_len, int32_t causal, int32_t window, void* out, float* lse, void* workspace,
                          size_t workspace_bytes, jgdpa_stream_t stream) {
  return fwd_impl(q, k, v, q_offsets, kv_offsets, batch, total_q, total_kv, heads, head_dim, act, scale,
                  bias_table, bias_len, causal, window, out, lse, workspace, workspace_bytes, stream);
}

}  // extern "C"

namespace {

// The backward; `ev` (3 caller events, entries may be null) is recorded on
// the stream before the dK/dV pass, between the passes and after the dQ pass.
jgdpa_status bwd_impl(const void* q, const void* k, const void* v, const void* out, const float* lse,
                      const void* dout, const int32_t* q_offsets, const int32_t* kv_offsets, int32_t batch,
                      int64_t total_q, int64_t total_kv, int32_t heads, int32_t head_dim, jgdpa_act act,
                      float scale, const float* bias_table, int32_t bias_len, int32_t causal, int32_t window,
                      void* dq, void* dk, void* dv, float* dbias, void* workspace, size_t workspace_bytes,
                      jgdpa_stream_t stream_, void* ds_scratch, size_t ds_scratch_bytes, void* const* ev,
                      int32_t q_shared = 0) {
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  auto record = [&](int i) -> cudaError_t {
    return (ev != nullptr && ev[i] != nullptr) ? cudaEventRecord(static_cast<cudaEvent_t>(ev[i]), stream)
                                               : cudaSuccess;
  };
  jgdpa_status st = check_common(batch, total_q, total_kv, heads, head_dim, act, scale, bias_table, bias_len,
                                 causal, q_shared > 0 ? kv_offsets : q_offsets, kv_offsets);
  if (st != JGDPA_OK) return st;
  if (window < 0) return JGDPA_ERR_INVALID_ARGUMENT;
  if (dbias != nullptr && bias_len == 0) return JGDPA_ERR_INVALID_ARGUMENT;
  if (total_q > 0 && (q == nullptr || dout == nullptr || dq == nullptr)) return JGDPA_ERR_INVALID_ARGUMENT;
  if (total_kv > 0 && (k == nullptr || v == nullptr || dk == nullptr || dv == nullptr))
    return JGDPA_ERR_INVALID_ARGUMENT;
  if (act == JGDPA_ACT_SOFTMAX && total_q > 0 && (out == nullptr || lse == nullptr))
    return JGDPA_ERR_INVALID_ARGUMENT;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16) || !aligned(dout, 16) ||
      !aligned(dq, 16) || !aligned(dk, 16) || !aligned(dv, 16) || !aligned(lse, 4) || !aligned(dbias, 4))
    return JGDPA_ERR_MISALIGNED;
  Layout L;
  if (!layout_for(batch, total_q, total_kv, heads, act, bias_len, true, &L, q_shared, head_dim))
    return JGDPA_ERR_CUDA;
  if (workspace == nullptr || workspace_bytes < L.total) return JGDPA_ERR_WORKSPACE_TOO_SMALL;
  if (!aligned(workspace, kAlign)) return JGDPA_ERR_MISALIGNED;
  // the fused dQ needs no stored dS: a scratch the caller passes is not used
  if (L.fused_dq) {
    ds_scratch = nullptr;
    ds_scratch_bytes = 0;
  }
  // stored dS: capacity in tiles (the device checks the lengths against it)
  const int64_t ds_tiles = ds_scratch ? static_cast<int64_t>(ds_scratch_bytes / jg::kDsTileBytes) : -1;
  if (ds_scratch && !aligned(ds_scratch, kAlign)) return JGDPA_ERR_MISALIGNED;
  if (ds_scratch && ds_tiles > INT32_MAX / jg::kTile) return JGDPA_ERR_UNSUPPORTED;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  JG_CUDA(cudaMemsetAsync(ws + L.header, 0, 64 * sizeof(int), stream));
  if (dbias) JG_CUDA(cudaMemsetAsync(dbias, 0, static_cast<size_t>(heads) * bias_len * sizeof(float), stream));
  if (batch == 0) return JGDPA_OK;
  const size_t row_bytes = static_cast<size_t>(heads) * head_dim * 2;
  const int64_t dq_rows = q_shared > 0 ? q_shared : total_q;  // rows of dq
  if (total_q == 0 || total_kv == 0) {  // no valid pair anywhere: all gradients are zero
    if (total_q) JG_CUDA(cudaMemsetAsync(dq, 0, dq_rows * row_bytes, stream));
    if (total_kv) {
      JG_CUDA(cudaMemsetAsync(dk, 0, total_kv * row_bytes, stream));
      JG_CUDA(cudaMemsetAsync(dv, 0, total_kv * row_bytes, stream));
    }
    return JGDPA_OK;
  }
  const bool stored_ds = ds_scratch != nullptr && ds_tiles > 0;
  if (q_shared > 0) {
    int32_t* qo = reinterpret_cast<int32_t*>(ws + L.q_off);
    shared_q_offsets_kernel<<<static_cast<unsigned>((batch + 1 + 255) / 256), 256, 0, stream>>>(qo, batch, q_shared);
    JG_CUDA(cudaGetLastError());
    q_offsets = qo;
  }
  const bool shortq = shortq_bwd_applies(q_shared, act);
  // (a scratch smaller than one tile is no scratch: every dQ is recomputed)
  // every backward but the fused-dQ ones forms the dQ of single-key-tile
  // segments in its key-major pass
  const bool dq_direct = !L.fused_dq && window == 0;
  st = run_sched(q_offsets, kv_offsets, batch, heads, total_q, total_kv, causal, window, ws, L, true, stream,
                 stored_ds ? ds_tiles : -1, shortq, dq_direct);
  if (st != JGDPA_OK) return st;

  jg::BwdParams p{};
  // the short-query backward loads its query and dO blocks as boxes of its
  // block width (16, 32 or 64 rows)
  const int q_box = shortq ? (q_shared <= 16 ? 16 : (q_shared <= 32 ? 32 : 64)) : kTile;
  if (!make_map(&p.tm_q, q, dq_rows, heads, head_dim, q_box) || !make_map(&p.tm_k, k, total_kv, heads, head_dim) ||
      !make_map(&p.tm_v, v, total_kv, heads, head_dim) ||
      !make_map(&p.tm_do, dout, total_q, heads, head_dim, q_box))
    return JGDPA_ERR_CUDA;
  p.q_shared = q_shared > 0 ? 1 : 0;
  p.dq_part = (q_shared > 0 && !L.fused_dq) ? reinterpret_cast<float*>(ws + L.dq_part) : nullptr;
  if (L.fused_dq) {
    p.dq_fused = reinterpret_cast<float*>(ws + L.dq_fused);
    p.kv_item_base = reinterpret_cast<const int32_t*>(ws + L.item_base);  // list 0: the key tiles
    p.q_rows = q_shared;
  }
  // direct dQ at d = 128 (into dq): TMA stores of 32-row blocks
  if (dq_direct && q_shared == 0 && !make_map(&p.tm_dq, dq, total_q, heads, head_dim, 32)) return JGDPA_ERR_CUDA;
  if (stored_ds) {
    if (!make_ds_map(&p.tm_ds, ds_scratch, ds_tiles)) return JGDPA_ERR_CUDA;
    p.ds_base = reinterpret_cast<const int64_t*>(ws + L.ds_base);
  }
  int* hdr = reinterpret_cast<int*>(ws + L.header);
  p.q_off = q_offsets;
  p.kv_off = kv_offsets;
  p.status = hdr;
  p.bias = bias_table;
  p.lse = lse;
  p.delta = act == JGDPA_ACT_SOFTMAX ? reinterpret_cast<float*>(ws + L.delta) : nullptr;
  p.dq = static_cast<__nv_bfloat16*>(dq);
  p.dk = static_cast<__nv_bfloat16*>(dk);
  p.dv = static_cast<__nv_bfloat16*>(dv);
  p.total_q = total_q;
  p.heads = heads;
  p.bias_len = bias_len;
  p.causal = causal;
  p.window = window;
  p.scale = scale;
  p.wait_limit_ns = wait_limit_ns();
  if (act == JGDPA_ACT_SOFTMAX)
    JG_CUDA(jg::launch_softmax_delta(out, dout, const_cast<float*>(p.delta), total_q, heads, head_dim, hdr,
                                     stream));
  const int grid_kv = static_cast<int>(std::min<int64_t>(L.grid, std::max(1, L.max0)));
  const int grid_q = static_cast<int>(std::min<int64_t>(L.grid, std::max(1, L.max1)));
  auto* part = dbias ? reinterpret_cast<unsigned long long*>(ws + L.dbias) : nullptr;
  if (part)
    JG_CUDA(cudaMemsetAsync(part, 0, static_cast<size_t>(grid_kv) * heads * bias_len * sizeof(*part), stream));
  p.dbias_part = part;
  p.units = reinterpret_cast<const jg::Unit*>(ws + L.units0);
  p.n_units = hdr + 1;
  JG_CUDA(record(0));
  if (shortq) JG_CUDA(jg::launch_bwd_shortq(p, head_dim, act, q_shared, grid_kv, stream));
  else JG_CUDA(jg::launch_bwd_pass(p, head_dim, act, true, grid_kv, stream));
  if (dq_direct) {  // the segments with one key tile: dK, dV and dQ in one pass
    p.units = reinterpret_cast<const jg::Unit*>(ws + L.units3);
    p.n_units = hdr + 4;
    JG_CUDA(jg::launch_bwd_pass(p, head_dim, act, true, grid_kv, stream, true));
  }
  JG_CUDA(record(1));
  p.dbias_part = nullptr;
  p.units = reinterpret_cast<const jg::Unit*>(ws + L.units1);
  p.n_units = hdr + 2;
  if (L.fused_dq) {  // dQ = the ordered sum of the key-major pass's contributions
    JG_CUDA(jg::launch_dq_fused_reduce(p.dq_fused, reinterpret_cast<float*>(ws + L.dq_fused_tmp), dq,
                                       p.kv_item_base, batch, heads, q_shared, head_dim, hdr, stream));
  } else if (stored_ds) {
    // dQ from the stored tiles for the segments that fit the scratch, then by
    // recomputation for the rest (a pass with an empty list ends at once)
    JG_CUDA(jg::launch_dq_ds(p, head_dim, grid_q, stream));
    p.units = reinterpret_cast<const jg::Unit*>(ws + L.units2);
    p.n_units = hdr + 3;
    JG_CUDA(jg::launch_bwd_pass(p, head_dim, act, false, grid_q, stream));
  } else {
    JG_CUDA(jg::launch_bwd_pass(p, head_dim, act, false, grid_q, stream));
  }
  JG_CUDA(record(2));
  if (part) JG_CUDA(jg::launch_dbias_reduce(part, dbias, grid_kv, heads * bias_len, stream));
  if (q_shared > 0 && !L.fused_dq)
    JG_CUDA(jg::launch_dq_shared_reduce(p.dq_part, dq, batch, static_cast<int64_t>(q_shared) * heads * head_dim, hdr,
                                        stream));
  return JGDPA_OK;
}

}  // namespace

extern "C" {

jgdpa_status jgdpa_bwd(const void* q, const void* k, const void* v, const void* out, const float* lse,
                       const void* dout, const int32_t* q_offsets, const int32_t* kv_offsets, int32_t batch,
                       int64_t total_q, int64_t total_kv, int32_t heads, int32_t head_dim, jgdpa_act act,
                       float scale, const float* bias_table, int32_t bias_len, int32_t causal, void* dq, void* dk,
                       void* dv, float* dbias, void* workspace, size_t workspace_bytes, jgdpa_stream_t stream) {
  return bwd_impl(q, k, v, out, lse, dout, q_offsets, kv_offsets, batch, total_q, total_kv, heads, head_dim, act,
                  scale, bias_table, bias_len, causal, 0, dq, dk, dv, dbias, workspace, workspace_bytes, stream,
                  nullptr, 0, nullptr);
}

jgdpa_status jgdpa_bwd_ex(const void* q, const void* k, const void* v, const void* out, const float* lse,
                          const void* dout, const int32_t* q_offsets, const int32_t* kv_offsets, int32_t batch,
                          int64_t total_q, int64_t total_kv, int32_t heads, int32_t head_dim, jgdpa_act act,
                          float scale, const float* bias_table, int32_t bias_len, int32_t causal,
                          int32_t window, void* dq, void* dk, void* dv, float* dbias, void* workspace,
                          size_t workspace_bytes, void* ds_scratch, size_t ds_scratch_bytes, jgdpa_stream_t stream,
                          void* const* pass_events) {
  return bwd_impl(q, k, v, out, lse, dout, q_offsets, kv_offsets, batch, total_q, total_kv, heads, head_dim, act,
                  scale, bias_table, bias_len, causal, window, dq, dk, dv, dbias, workspace, workspace_bytes,
                  stream, ds_scratch, ds_scratch_bytes, pass_events);
}

size_t jgdpa_shared_q_workspace_bytes(int32_t batch, int32_t n_shared, int64_t total_kv, int32_t heads,
                                      int32_t head_dim, jgdpa_act act, int32_t bias_len, int32_t for_backward) {
  if (batch < 0 || n_shared < 1 || total_kv < 0 || heads < 1 || bias_len < 0) return 0;
  if (head_dim != 32 && head_dim != 64 && head_dim != 128) return 0;
  const int64_t total_q = static_cast<int64_t>(batch) * n_shared;
  if (total_q > INT32_MAX) return 0;
  Layout L;
  if (!layout_for(batch, total_q, total_kv, heads, act, bias_len, for_backward != 0, &L, n_shared, head_dim))
    return 0;
  return L.total;
}

jgdpa_status jgdpa_fwd_shared_q(const void* q, int32_t n_shared, const void* k, const void* v,
                                const int32_t* kv_offsets, int32_t batch, int64_t total_kv, int32_t heads,
                                int32_t head_dim, jgdpa_act act, float scale, const float* bias_table,
                                int32_t bias_len, int32_t causal, int32_t window, void* out, float* lse,
                                void* workspace, size_t workspace_bytes, jgdpa_stream_t stream) {
  if (n_shared < 1 || batch < 0) return JGDPA_ERR_INVALID_ARGUMENT;
  const int64_t total_q = static_cast<int64_t>(batch) * n_shared;
  if (total_q > INT32_MAX) return JGDPA_ERR_UNSUPPORTED;
  return fwd_impl(q, k, v, nullptr, kv_offsets, batch, total_q, total_kv, heads, head_dim, act, scale, bias_table,
                  bias_len, causal, window, out, lse, workspace, workspace_bytes, stream, n_shared);
}

jgdpa_status jgdpa_bwd_shared_q(const void* q, int32_t n_shared, const void* k, const void* v, const void* out,
                                const float* lse, const void* dout, const int32_t* kv_offsets, int32_t batch,
                                int64_t total_kv, int32_t heads, int32_t head_dim, jgdpa_act act, float scale,
                                const float* bias_table, int32_t bias_len, int32_t causal, int32_t window,
                                void* dq, void* dk, void* dv, float* dbias, void* workspace,
                                size_t workspace_bytes, void* ds_scratch, size_t ds_scratch_bytes,
                                jgdpa_stream_t stream, void* const* pass_events) {
  if (n_shared < 1 || batch < 0) return JGDPA_ERR_INVALID_ARGUMENT;
  const int64_t total_q = static_cast<int64_t>(batch) * n_shared;
  if (total_q > INT32_MAX) return JGDPA_ERR_UNSUPPORTED;
  return bwd_impl(q, k, v, out, lse, dout, nullptr, kv_offsets, batch, total_q, total_kv, heads, head_dim, act,
                  scale, bias_table, bias_len, causal, window, dq, dk, dv, dbias, workspace, workspace_bytes,
                  stream, ds_scratch, ds_scratch_bytes, pass_events, n_shared);
}

size_t jgdpa_ds_scratch_bytes(const int32_t* q_offsets_host, const int32_t* kv_offsets_host, int32_t batch,
                              int32_t heads, int32_t window) {
  if (batch < 0 || heads < 1 || window < 0 ||
      (batch > 0 && (q_offsets_host == nullptr || kv_offsets_host == nullptr)))
    return 0;
  uint64_t tiles = 0;
  for (int32_t b = 0; b < batch; ++b) {
    const int64_t lq = static_cast<int64_t>(q_offsets_host[b + 1]) - q_offsets_host[b];
    const int64_t lkv = static_cast<int64_t>(kv_offsets_host[b + 1]) - kv_offsets_host[b];
    if (lq < 0 || lkv < 0) return 0;
    // (a segment whose dQ the key-major pass forms directly stores nothing)
    if (jg::dq_direct_segment(static_cast<int>(lq), static_cast<int>(lkv), window)) continue;
    const int64_t nq = (lq + jg::kTile - 1) / jg::kTile, nk = (lkv + jg::kTile - 1) / jg::kTile;
    tiles += static_cast<uint64_t>(nk) * static_cast<uint64_t>(jg::ds_span(nq, window));
  }
  return static_cast<size_t>(tiles * heads * jg::kDsTileBytes);
}

jgdpa_status jgdpa_read_device_status(const void* workspace, jgdpa_stream_t stream_) {
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  if (workspace == nullptr) return JGDPA_ERR_INVALID_ARGUMENT;
  int s = 0;
  if (cudaMemcpyAsync(&s, workspace, sizeof(int), cudaMemcpyDeviceToHost, stream) != cudaSuccess)
    return JGDPA_ERR_CUDA;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return JGDPA_ERR_CUDA;
  return static_cast<jgdpa_status>(s);
}

const char* jgdpa_status_string(jgdpa_status s) {
  switch (s) {
    case JGDPA_OK: return "ok";
    case JGDPA_ERR_INVALID_ARGUMENT: return "invalid argument";
    case JGDPA_ERR_UNSUPPORTED: return "unsupported configuration";
    case JGDPA_ERR_MISALIGNED: return "misaligned pointer";
    case JGDPA_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case JGDPA_ERR_CUDA: return "CUDA error";
    case JGDPA_ERR_BAD_OFFSETS: return "bad offsets (device-detected)";
    case JGDPA_ERR_DEVICE_TIMEOUT: return "device wait timed out";
  }
  return "unknown status";
}

void jgdpa_set_wait_limit_ns(uint64_t limit_ns) { g_wait_limit_ns.store(limit_ns, std::memory_order_relaxed); }

jgdpa_status jgdpa_eval_activation(jgdpa_act act, int32_t path, const float* x, int64_t n, float* y, float* dy,
                                   jgdpa_stream_t stream_) {
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  if ((act != JGDPA_ACT_GELU && act != JGDPA_ACT_SILU) || path < 0 || path > 2 || n < 0)
    return JGDPA_ERR_INVALID_ARGUMENT;
  if (n == 0) return JGDPA_OK;
  if (x == nullptr || y == nullptr) return JGDPA_ERR_INVALID_ARGUMENT;
  eval_act_kernel<<<static_cast<unsigned>((n + 511) / 512), 256, 0, stream>>>(act, path, x, n, y, dy);
  JG_CUDA(cudaGetLastError());
  return JGDPA_OK;
}

}  // extern "C"

// --------------------------------------------------------------------------
// Forward without a caller workspace: scratch lives in a fixed device array.
namespace {

__device__ __align__(256) uint8_t g_noalloc_scratch[JGDPA_NOALLOC_SCRATCH_BYTES];

std::mutex g_noalloc_mu;
void* g_noalloc_addr[128] = {};

// Device address of g_noalloc_scratch on the current device, looked up once
// per device with that device current.  (In host code the array's name is
// only a host-side stand-in and must never reach a kernel.)
jgdpa_status noalloc_scratch(void** addr) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return JGDPA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (g_noalloc_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return JGDPA_ERR_CUDA;
    g_noalloc_addr[dev] = p;
  }
  *addr = g_noalloc_addr[dev];
  return JGDPA_OK;
}

}  // namespace

extern "C" jgdpa_status jgdpa_fwd_noalloc(const void* q, const void* k, const void* v, const int32_t* q_offsets,
                                          const int32_t* kv_offsets, int32_t batch, int64_t total_q,
                                          int64_t total_kv, int32_t heads, int32_t head_dim, jgdpa_act act,
                                          float scale, const float* bias_table, int32_t bias_len, int32_t causal,
                                          void* out, float* lse, jgdpa_stream_t stream) {
  jgdpa_status st = check_common(batch, total_q, total_kv, heads, head_dim, act, scale, bias_table, bias_len,
                                 causal, q_offsets, kv_offsets);
  if (st != JGDPA_OK) return st;
  Layout L;
  if (!layout_for(batch, total_q, total_kv, heads, act, bias_len, false, &L)) return JGDPA_ERR_CUDA;
  if (L.total > JGDPA_NOALLOC_SCRATCH_BYTES) return JGDPA_ERR_WORKSPACE_TOO_SMALL;
  void* scratch = nullptr;
  st = noalloc_scratch(&scratch);
  if (st != JGDPA_OK) return st;
  return fwd_impl(q, k, v, q_offsets, kv_offsets, batch, total_q, total_kv, heads, head_dim, act, scale,
                  bias_table, bias_len, causal, 0, out, lse, scratch, JGDPA_NOALLOC_SCRATCH_BYTES, stream);
}
