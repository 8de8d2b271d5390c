// Parameters and small helpers shared by the GDPA kernels and their launcher.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

namespace jg {

constexpr int kTile = 128;          // rows per Q / K / V tile (= MMA M and N)
constexpr int kMaxBiasLen = 4095;   // largest accepted bias table (2R + 1)
constexpr int kCostBuckets = 4096;  // scheduler's counting-sort buckets

// Kinds of work lists built by the scheduler.
enum UnitKind : int {
  kUnitsFwd = 0,   // (segment, head, pair of 128-row query tiles)
  kUnitsKv = 1,    // (segment, head, 128-row key/value tile): dK, dV
  kUnitsQ = 2,     // (segment, head, 128-row query tile): dQ
  // With a stored-dS scratch: the query-tile units of the segments whose dS
  // tiles fit the scratch (dQ from the stored tiles) and of the others (dQ by
  // recomputation).  A segment's tiles fit when the prefix of the tile counts
  // up to and including it is within the scratch's capacity.
  kUnitsQStored = 3,
  kUnitsQRecompute = 4,
  // Short-query backward: (segment, head, chunk of up to kChunkTiles key
  // tiles); z = the chunk index.
  kUnitsKvChunk = 5,
  // Key-major units of the segments whose dQ the key-major pass forms
  // directly (dq_direct_segment); kUnitsKv then holds the others.
  kUnitsKvDirect = 6,
  // Forward units (segment, head, chunk of up to kChunkTiles query tiles) of
  // the segments with kv_resident_segment; kUnitsFwd then holds the others.
  kUnitsFwdKvRes = 7,
};
constexpr int kChunkTiles = 16;

// One work unit: x = segment, y = head, z = tile (or tile pair) index, w = cost.
using Unit = int4;

struct SchedList {
  int kind;
  int max_units;
  int* n_units;   // device counter written by the scheduler
  Unit* units;    // device list, longest first
};

struct SchedParams {
  const int32_t* q_off;
  const int32_t* kv_off;
  int32_t batch;
  int32_t heads;
  int64_t total_q;
  int64_t total_kv;
  int32_t causal;
  int32_t window;       // > 0: sliding window |i - j| < window
  int* status;
  int32_t* item_base;   // scratch [batch + 1] per list
  SchedList list[4];
  int n_lists;
  // backward with stored dS: first dS tile of each segment, or -1 for a
  // segment whose tiles do not fit ([batch + 1]; entry batch = tiles used);
  // nullptr without a scratch
  int64_t* ds_base;
  int64_t ds_capacity;  // dS tiles the caller's scratch holds
  // Segments whose keys fit one tile get their own lists: in the forward
  // those with kv_resident_segment go to kUnitsFwdKvRes; in the backward
  // those with dq_direct_segment go to kUnitsKvDirect and get no query-major
  // units and no stored dS.
  int32_t one_tile;
};

// Lengths and tile counts of one segment.
struct Seg {
  int q0, lq, k0, lkv;
};

__device__ __forceinline__ Seg load_seg(const int32_t* q_off, const int32_t* kv_off, int b) {
  Seg s;
  s.q0 = __ldg(q_off + b);
  s.lq = __ldg(q_off + b + 1) - s.q0;
  s.k0 = __ldg(kv_off + b);
  s.lkv = __ldg(kv_off + b + 1) - s.k0;
  return s;
}

__host__ __device__ __forceinline__ int ceil_div(int a, int b) { return (a + b - 1) / b; }

// The partner tiles [first, first + count) that one 128-row tile meets.
// Query row i and key row j (segment-local) form a pair when j < Lkv and,
// with top-left causal masking, j <= i, and with a sliding window w > 0,
// |i - j| < w.
struct TileSpan {
  int first, count;
};

// Rows [128 t, 128 t + 127] reach partner rows [128 t - (w - 1), 128 t + 127 + (w - 1)].
__device__ __forceinline__ void window_tiles(int t, int window, int& lo, int& hi) {
  if (window <= 0) return;
  const int64_t a = static_cast<int64_t>(t) * kTile - (window - 1);
  const int64_t b = static_cast<int64_t>(t) * kTile + (kTile - 1) + (window - 1);
  lo = max(lo, a <= 0 ? 0 : static_cast<int>(a / kTile));
  hi = static_cast<int>(min(static_cast<int64_t>(hi), b / kTile + 1));
}
// Key/value tiles that query tile t visits (causal: tiles 0..t at most).
__device__ __forceinline__ TileSpan kv_span_for_q_tile(int t, int lkv, int causal, int window) {
  int lo = 0, hi = ceil_div(lkv, kTile);
  if (causal) hi = min(hi, t + 1);
  window_tiles(t, window, lo, hi);
  return {lo, max(0, hi - lo)};
}
// Query tiles that key/value tile kt meets (causal: tiles kt.. at least).
__device__ __forceinline__ TileSpan q_span_for_kv_tile(int kt, int lq, int causal, int window) {
  int lo = causal ? kt : 0, hi = ceil_div(lq, kTile);
  window_tiles(kt, window, lo, hi);
  return {lo, max(0, hi - lo)};
}

// A segment whose keys fit one tile: the key-major backward forms each query
// tile's dQ itself (dS K with that key tile, complete after one product), so
// the segment needs no stored dS and no query-major dQ units.
// (Without a window only: under a window the single key tile may not reach
// every query tile.)
__host__ __device__ __forceinline__ bool dq_direct_segment(int lq, int lkv, int window) {
  return window <= 0 && lq > 0 && lkv > 0 && lkv <= kTile;
}

// Forward: a segment whose keys fit one tile runs in the key/value-resident
// forward (K and V loaded once for up to kChunkTiles query tiles).  Segments
// of a single query tile share nothing there, but taking them too leaves the
// general forward fewer units, often none, when keys are short: measured
// -1.4% on the short-K/V forward, no change on causal softmax.
__host__ __device__ __forceinline__ bool kv_resident_segment(int lq, int lkv, int window) {
  return dq_direct_segment(lq, lkv, window);
}

// Index of the i-th unit processed by CTA c of G (serpentine over rounds, so
// that each round's longest units are spread evenly).
__device__ __forceinline__ int unit_index(int round, int c, int g) {
  return round * g + ((round & 1) ? (g - 1 - c) : c);
}

struct FwdParams {
  CUtensorMap tm_q;
  CUtensorMap tm_k;
  CUtensorMap tm_v;
  const int32_t* q_off;
  const int32_t* kv_off;
  const Unit* units;
  const int* n_units;
  int* status;
  const float* bias;      // [H][bias_len] or nullptr
  __nv_bfloat16* out;     // [total_q][H][D]
  float* lse;             // [H][total_q] (softmax) or nullptr
  int64_t total_q;
  int32_t heads;
  int32_t bias_len;
  int32_t causal;
  int32_t window;         // > 0: sliding window |i - j| < window
  float scale;            // s (GELU/SiLU) or s * log2(e) (softmax)
  unsigned long long wait_limit_ns;  // limit of one internal wait
  int32_t q_shared;       // 1: every segment reads the same query rows (Q map row 0 = its row 0)
  // the key/value-resident forward's O stores: boxes of 32 rows x 1 head x
  // min(d, 64) columns over out, 128-byte swizzle (d >= 64, GELU / SiLU)
  CUtensorMap tm_o;
};

struct BwdParams {
  CUtensorMap tm_q;
  CUtensorMap tm_k;
  CUtensorMap tm_v;
  CUtensorMap tm_do;
  const int32_t* q_off;
  const int32_t* kv_off;
  const Unit* units;
  const int* n_units;
  int* status;
  const float* bias;       // [H][bias_len] or nullptr
  const float* lse;        // [H][total_q] (softmax)
  const float* delta;      // [H][total_q] rowsum(dO * O) (softmax)
  __nv_bfloat16* dq;
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  unsigned long long* dbias_part;  // [gridDim.x][H][bias_len] per-CTA fixed-point partial sums, or nullptr
  int64_t total_q;
  int32_t heads;
  int32_t bias_len;
  int32_t causal;
  int32_t window;          // > 0: sliding window |i - j| < window
  float scale;             // s
  // Stored dS (optional): the dK/dV pass writes every bf16 dS^T tile to a
  // scratch array of [128 keys][128 queries] tiles; tile of (segment b, head
  // h, key tile kt, query tile qt) = ds_base[b] + (h nk_b + kt) span_b +
  // slot (see ds_span / ds_slot).
  CUtensorMap tm_ds;       // 2-D over the scratch: 128 columns x (tiles * 128) rows
  const int64_t* ds_base;  // nullptr: no stored dS; entry < 0: that segment's dS is not stored
  unsigned long long wait_limit_ns;  // limit of one internal wait
  int32_t q_shared;        // 1: every segment reads the same query rows (Q map row 0 = its row 0)
  float* dq_part;          // q_shared: fp32 dQ of every segment's rows [total_q][H][D], summed afterwards
  // Fused dQ (shared queries with at most 128 rows, d <= 64): the key-major
  // pass also forms each unit's dQ contribution dS K and writes it in fp32 to
  // dq_fused[(kv_item_base[b] + kt) H + h][q_rows][D]; no dS is stored and no
  // dQ pass runs.  nullptr otherwise.
  float* dq_fused;
  const int32_t* kv_item_base;  // the scheduler's key-tile prefix per segment
  int32_t q_rows;               // rows of each dq_fused block (the shared query count)
  // direct dQ at d = 128: boxes of 32 rows x 1 head x 64 columns over dq,
  // 128-byte swizzle (the X tile's layout), for the TMA stores of dQ
  CUtensorMap tm_dq;
};

constexpr int kDsTileBytes = kTile * kTile * 2;

// Host side: a kernel's dynamic shared-memory limit is a per-device
// attribute; each launcher keeps, per kernel, one flag per device and sets
// the attribute only the first time it launches that kernel on a device.
constexpr int kMaxDevices = 128;
using DeviceFlags = std::atomic<unsigned char>[kMaxDevices];
template <typename Kernel>
inline cudaError_t smem_attr_once(Kernel kern, int bytes, DeviceFlags& done) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const bool cached = dev >= 0 && dev < kMaxDevices;
  if (cached && done[dev].load(std::memory_order_acquire)) return cudaSuccess;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && cached) done[dev].store(1, std::memory_order_release);
  return e;
}

// dbias partial sums are 64-bit two's-complement fixed point with this many
// fraction bits (resolution 2^-24, range +-2^39).  Integer additions are exact
// and commute, so the sums do not depend on the order in which the CTAs' warps
// add their contributions or on which CTA ran which unit: dbias is the same
// bit for bit on every run.
constexpr int kDbiasFracBits = 24;
__device__ __forceinline__ unsigned long long dbias_fixed(float v) {
  return static_cast<unsigned long long>(__float2ll_rn(v * static_cast<float>(1 << kDbiasFracBits)));
}

// Stored-dS slots per key tile of a segment with nq query tiles: nq, or
// under a window short enough to pay, the 2e + 1 query tiles kt - e .. kt + e
// that key tile kt can meet (e = ceil((w - 1) / 128)); the slot of query
// tile qt is then qt - kt + e.
__host__ __device__ __forceinline__ int64_t ds_band_reach(int window) {
  return (static_cast<int64_t>(window) + kTile - 2) / kTile;
}
__host__ __device__ __forceinline__ int64_t ds_span(int64_t nq, int window) {
  if (window <= 0) return nq;
  const int64_t band = 2 * ds_band_reach(window) + 1;
  return band < nq ? band : nq;
}
__device__ __forceinline__ int64_t ds_slot(int64_t nq, int window, int kt, int qt) {
  if (window <= 0 || ds_span(nq, window) == nq) return qt;
  return qt - kt + ds_band_reach(window);
}

// First row of a dS tile in the scratch's 2-D view.
__device__ __forceinline__ int ds_row(const int64_t* ds_base, const Seg& s, int b, int h, int kt, int qt,
                                      int window) {
  const int64_t nq = ceil_div(s.lq, kTile), nk = ceil_div(s.lkv, kTile);
  const int64_t span = ds_span(nq, window);
  return static_cast<int>(
      (__ldg(ds_base + b) + (static_cast<int64_t>(h) * nk + kt) * span + ds_slot(nq, window, kt, qt)) * kTile);
}

}  // namespace jg
