// Backward jagged GDPA kernels for sm_103a.
//
// The backward is split in two persistent passes so that every output tile
// has exactly one writer and no atomics touch dQ, dK or dV (the split-dQ,
// atomics-free backward of "Eliminating Compute Waste in Asymmetric
// Workloads", aiuniverse.news):
//
//   dkdv pass, unit = (segment, head, 128-row key/value tile):
//     for every query tile i that meets it:
//       S^T = K Q^T, dP^T = V dO^T                       (tcgen05, TMEM)
//       phase A: P^T = act(x)^T (bf16, into TMEM over S^T), act'(x) kept
//                in registers (softmax: P = exp(x - LSE_i))
//       phase B: dS^T = dP^T act'(x)^T (softmax: P (dP - D_i)), to shared
//                memory; dbias partial sums
//       dV += P^T dO, dK += dS^T Q                       (tcgen05, TMEM)
//     dK *= s; store dK, dV
//   dq pass, unit = (segment, head, 128-row query tile):
//     for every key/value tile: S = Q K^T, dP = dO V^T,
//       phase A: act'(x); phase B: dS = dP act'(x) to shared memory;
//       dQ += dS K
//     dQ *= s; store
//
// The bf16 dS^T / dS that the activation warps produce go to a shared "X"
// tile, where the dK / dQ products, the TMA store of the dS tiles and the
// direct dQ product read them.  In dkdv only one X tile fits at d = 128, and
// P^T and dS^T sharing it serialised phase B behind dV; P^T goes back into
// TMEM over S^T instead, and dV reads it from there -- which is also the
// faster form: on this GPU an MMA whose A operand is in TMEM reads only B
// from shared memory, and a 128 x 128 x 16 product takes ~80 cycles that way
// against ~110 with both operands in shared memory (the shared-memory
// operand stream, ~73 bytes a clock, is the limit).  The activation warps
// load a whole S (dP) tile into registers before computing, so the next
// tile's S (dP) is computed while they work.
//
// TMEM (512 columns): dkdv uses S^T [0,128), dP^T [128,256), dV [256,256+D),
// dK [256+D, 256+2D); dq uses S [0,128), dP [128,256), dQ [256,256+D).  Two
// activation warpgroups split the 128 columns of a tile; warpgroup h owns
// columns [64h, 64h + 64), which is column block h of the X tile.
#include "act.cuh"
#include "common.cuh"
#include "ptx.cuh"

namespace jg {

// Number of the four 16-column groups that each activation thread owns per
// tile whose act / act' take the ALU route (the rest use the
// special-function unit).  Measured on GB300 (long-tail workload, d = 128,
// GELU): 0/1/2 groups gave a dK/dV pass of 5.68/6.26/6.90 ms, so 0 is the
// default and the route a compile-time option.
#ifndef JGDPA_BWD_ALU_GROUPS
#define JGDPA_BWD_ALU_GROUPS 0
#endif
constexpr int kBwdAluGroups = JGDPA_BWD_ALU_GROUPS;

// Layout of one swizzled [128][D] bf16 tile in shared memory.
template <int D>
struct TileCfg {
  static constexpr int kBlockCols = D < 64 ? D : 64;
  static constexpr int kRowBytes = kBlockCols * 2;
  static constexpr int kBlockBytes = kTile * kRowBytes;
  static constexpr int kNumBlocks = D / kBlockCols;
  static constexpr int kTileBytes = kTile * D * 2;
  static constexpr uint32_t kSwizzle = kRowBytes == 128 ? 2u : 4u;
  static constexpr int kSBO = 8 * kRowBytes;
};

// Shared memory of one pass.  Resident pair: K, V (dkdv) or Q, dO (dq).
// Streamed operand A: Q (dkdv) or K (dq); streamed operand B: dO (dkdv) or
// V (dq); each has its own ring.  X: ring of [128][128] bf16 tiles written by
// the activation warps (P^T then dS^T per query tile in dkdv, dS in dq).
// Stage counts at d = 128 (seven 32 KB tiles fit): stream A (Q in dkdv, K in
// dq) is read at the start of a tile's life (S) and again at its end (dK /
// dQ), so it keeps three stages; stream B (dO / V) is read early (dP) and,
// in dkdv, once more by dV right after phase A, so one stage suffices; one X.
template <int D, bool KV_MAJOR>
struct BwdCfg : TileCfg<D> {
  using T = TileCfg<D>;
  static constexpr int kStagesA = D == 128 ? 3 : 4;
  static constexpr int kStagesB = D == 128 ? 1 : (D == 64 ? 2 : 4);
  static constexpr int kNumX = D == 128 ? 1 : 2;
  // resident pairs: two where they fit, so that the next unit's pair loads
  // while this one computes (units of one partner tile are otherwise
  // serialised on the copy latency)
  static constexpr int kNumRes = D == 128 ? 1 : 2;
  static constexpr int kXBytes = kTile * kTile * 2;
  static constexpr int kResOff = 0;
  static constexpr int kResBytes = 2 * T::kTileBytes;
  static constexpr int kAOff = kNumRes * kResBytes;
  static constexpr int kBOff = kAOff + kStagesA * T::kTileBytes;
  static constexpr int kXOff = kBOff + kStagesB * T::kTileBytes;
  static constexpr int kBarOff = kXOff + kNumX * kXBytes;
  static constexpr int kSmemBytes = kBarOff + 512 + 1024;
  static_assert(kXOff % 1024 == 0, "X tiles need 1024-byte alignment for the 128-byte swizzle");
  static_assert(kSmemBytes <= 232448, "shared memory per CTA");
};

struct BwdBars {
  uint64_t res_full[2], res_empty[2];
  uint64_t s_full, s_free, p_full, dp_full, dp_free, acc_full, acc_empty;
  uint64_t drain;
  uint64_t x_full[2], x_empty[2];
  uint64_t a_full[4], a_empty[4], b_full[4], b_empty[4];
  uint32_t tmem_base;
  int abort;
  uint64_t dq_full, dq_empty;  // direct dQ of one query tile (dK/dV pass, DIRECT kernels)
};

// K-major operand at column offset kk*16 inside a [128][D] tile: byte
// offset from the tile start (the descriptor's address field counts 16-byte
// units and never carries: shared addresses stay below 256 KB).
template <int D>
__host__ __device__ constexpr uint32_t kmajor_off(int kk) {
  using C = TileCfg<D>;
  return (kk * 16 / C::kBlockCols) * C::kBlockBytes + (kk * 16 % C::kBlockCols) * 2;
}
template <int D>
__device__ __forceinline__ uint64_t kmajor_desc0(uint32_t tile) {
  using C = TileCfg<D>;
  return sdesc(tile, 16, C::kSBO, C::kSwizzle);
}
// MN-major operand (N = D columns, K = 128 rows) at row offset kk*16.
template <int D>
__device__ __forceinline__ uint64_t mnmajor_desc0(uint32_t tile) {
  using C = TileCfg<D>;
  return sdesc(tile, C::kBlockBytes, C::kSBO, C::kSwizzle);
}

// C(tmem) = A_tile(128 x D) * B_tile(128 x D)^T : both K-major.  Called by
// the whole MMA warp; `leader` issues.
template <int D>
__device__ __forceinline__ void mma_tile_nt(uint32_t d_tmem, uint32_t a_tile, uint32_t b_tile, bool leader) {
  constexpr uint32_t idesc = idesc_bf16(kTile, kTile, 0, 0);
  const uint64_t a0 = kmajor_desc0<D>(a_tile), b0 = kmajor_desc0<D>(b_tile);
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint64_t off = kmajor_off<D>(kk) >> 4;
    if (leader) mma_ss(d_tmem, a0 + off, b0 + off, idesc, kk > 0 ? 1u : 0u);
  }
}
// C(tmem, 128 x D) (+)= X(128 x 128, K-major, 128-byte swizzle) * B_tile(128 x D, MN-major)
template <int D>
__device__ __forceinline__ void mma_tile_xs(uint32_t d_tmem, uint32_t x_tile, uint32_t b_tile, bool accumulate,
                                            bool leader) {
  using C = TileCfg<D>;
  constexpr uint32_t idesc = idesc_bf16(kTile, D, 0, 1);
  const uint64_t a0 = kmajor_desc0<kTile>(x_tile), b0 = mnmajor_desc0<D>(b_tile);
#pragma unroll
  for (int kk = 0; kk < kTile / 16; ++kk) {
    const uint64_t aoff = kmajor_off<kTile>(kk) >> 4;
    const uint64_t boff = static_cast<uint64_t>(kk * 16 * C::kRowBytes) >> 4;
    if (leader) mma_ss(d_tmem, a0 + aoff, b0 + boff, idesc, (accumulate || kk > 0) ? 1u : 0u);
  }
}

// C(tmem, 128 x D) (+)= A(tmem, 128 x 128 bf16: K steps 0-3 from a_lo, 4-7
// from a_hi) * B_tile(128 x D, MN-major)
template <int D>
__device__ __forceinline__ void mma_tile_ts(uint32_t d_tmem, uint32_t a_lo, uint32_t a_hi, uint32_t b_tile,
                                            bool accumulate, bool leader) {
  using C = TileCfg<D>;
  constexpr uint32_t idesc = idesc_bf16(kTile, D, 0, 1);
  const uint64_t b0 = mnmajor_desc0<D>(b_tile);
#pragma unroll
  for (int kk = 0; kk < kTile / 16; ++kk) {
    const uint32_t a = kk < 4 ? a_lo + kk * 8 : a_hi + (kk - 4) * 8;
    const uint64_t boff = static_cast<uint64_t>(kk * 16 * C::kRowBytes) >> 4;
    if (leader) mma_ts(d_tmem, a, b0 + boff, idesc, (accumulate || kk > 0) ? 1u : 0u);
  }
}

// C(tmem, 128 x D) = dS(128 x 128) * K(128 x D): the X tile (dS^T, K-major
// [keys][queries]) read as the MN-major A operand is dS, and the key tile
// ([keys][D], MN-major B) is K.
template <int D>
__device__ __forceinline__ void mma_ds_k(uint32_t d_tmem, uint32_t x_tile, uint32_t k_tile, bool leader) {
  using C = TileCfg<D>;
  constexpr uint32_t idesc = idesc_bf16(kTile, D, 1, 1);
  const uint64_t a0 = mnmajor_desc0<kTile>(x_tile), b0 = mnmajor_desc0<D>(k_tile);
#pragma unroll
  for (int kk = 0; kk < kTile / 16; ++kk) {
    const uint64_t aoff = static_cast<uint64_t>(kk * 16 * TileCfg<kTile>::kRowBytes) >> 4;
    const uint64_t boff = static_cast<uint64_t>(kk * 16 * C::kRowBytes) >> 4;
    if (leader) mma_ss(d_tmem, a0 + aoff, b0 + boff, idesc, kk > 0 ? 1u : 0u);
  }
}

// Unit geometry.  KV-major units: x = b, y = h, z = kv tile.  Q-major: z = q tile.
struct BwdUnit {
  int b, h, tile;
  Seg seg;
  int first;   // first partner tile
  int count;   // partner tiles visited
  int rows;    // valid rows of this unit's own tile
};

// WIN: the kernel is compiled for a sliding window (p.window > 0); the plain
// kernels fold the window away.
template <bool KV_MAJOR, bool WIN>
__device__ __forceinline__ BwdUnit bwd_unit(const BwdParams& p, int idx) {
  const int window = WIN ? p.window : 0;
  BwdUnit u;
  const Unit w = p.units[idx];
  u.b = w.x;
  u.h = w.y;
  u.tile = w.z;
  u.seg = load_seg(p.q_off, p.kv_off, u.b);
  if constexpr (!WIN) {  // the plain spans, written out (the general form measured ~1.4% slower in dK/dV)
    if constexpr (KV_MAJOR) {
      u.rows = u.seg.lkv - u.tile * kTile;
      u.first = p.causal ? u.tile : 0;
      const int n = ceil_div(u.seg.lq, kTile);
      u.count = p.causal ? max(0, n - u.tile) : n;
    } else {
      u.rows = u.seg.lq - u.tile * kTile;
      u.first = 0;
      const int n = ceil_div(u.seg.lkv, kTile);
      u.count = p.causal ? min(u.tile + 1, n) : n;
    }
    return u;
  }
  const TileSpan sp = KV_MAJOR ? q_span_for_kv_tile(u.tile, u.seg.lq, p.causal, window)
                               : kv_span_for_q_tile(u.tile, u.seg.lkv, p.causal, window);
  u.rows = (KV_MAJOR ? u.seg.lkv : u.seg.lq) - u.tile * kTile;
  u.first = sp.first;
  u.count = sp.count;
  return u;
}

// ----------------------------------------------------------------- producer
// Resident pair: (K, V) of the unit (dkdv) or (Q, dO) (dq).  Streamed pairs:
// (Q, dO) of each query tile (dkdv) or (K, V) of each key tile (dq).  Two
// producer threads: STREAM 0 loads the resident pair and stream A, STREAM 1
// stream B, so that a full ring of one stream never holds up the other.
template <int D, bool KV_MAJOR, int STREAM, bool WIN>
__device__ void bwd_producer(const BwdParams& p, uint8_t* smem, BwdBars* bars, int n_units, Fail fail) {
  using C = BwdCfg<D, KV_MAJOR>;
  constexpr int kStages = STREAM == 0 ? C::kStagesA : C::kStagesB;
  const CUtensorMap* res0 = KV_MAJOR ? &p.tm_k : &p.tm_q;
  const CUtensorMap* res1 = KV_MAJOR ? &p.tm_v : &p.tm_do;
  const CUtensorMap* str = STREAM == 0 ? (KV_MAJOR ? &p.tm_q : &p.tm_k) : (KV_MAJOR ? &p.tm_do : &p.tm_v);
  uint64_t* full = STREAM == 0 ? bars->a_full : bars->b_full;
  uint64_t* empty = STREAM == 0 ? bars->a_empty : bars->b_empty;
  uint8_t* ring = smem + (STREAM == 0 ? C::kAOff : C::kBOff);
  uint32_t res_it = 0, st_it = 0;
  const bool leader = elect_one();
  bool ok = true;
  for (int r = 0; ok; ++r) {
    const int idx = unit_index(r, blockIdx.x, gridDim.x);
    if (idx >= n_units) break;
    const BwdUnit u = bwd_unit<KV_MAJOR, WIN>(p, idx);
    if (u.count == 0) continue;
    if constexpr (STREAM == 0) {
      const int rs = res_it % C::kNumRes;
      if (!(ok = mbar_wait_warp(&bars->res_empty[rs], ((res_it / C::kNumRes) & 1) ^ 1, fail))) break;
      ++res_it;
      const int row = (KV_MAJOR ? u.seg.k0 : u.seg.q0) + u.tile * kTile;
      // shared queries (Q-major pass): the Q map holds the shared rows once
      const int row0 = (!KV_MAJOR && p.q_shared) ? u.tile * kTile : row;
      if (leader) {
        uint64_t* bar = &bars->res_full[rs];
        mbar_arrive_tx(bar, 2 * C::kTileBytes);
        uint8_t* d0 = smem + C::kResOff + rs * C::kResBytes;
#pragma unroll
        for (int cb = 0; cb < C::kNumBlocks; ++cb) {
          tma_load_3d(d0 + cb * C::kBlockBytes, res0, bar, cb * C::kBlockCols, u.h, row0);
          tma_load_3d(d0 + C::kTileBytes + cb * C::kBlockBytes, res1, bar, cb * C::kBlockCols, u.h, row);
        }
      }
    }
    // shared queries (key-major pass, stream A = Q): the Q map holds the shared rows once
    const int sbase = KV_MAJOR ? ((STREAM == 0 && p.q_shared) ? 0 : u.seg.q0) : u.seg.k0;
    for (int i = 0; i < u.count; ++i) {
      const int row = sbase + (u.first + i) * kTile;
      const int st = st_it % kStages;
      if (!(ok = mbar_wait_warp(&empty[st], ((st_it / kStages) & 1) ^ 1, fail))) break;
      if (leader) {
        mbar_arrive_tx(&full[st], C::kTileBytes);
        uint8_t* dst = ring + st * C::kTileBytes;
#pragma unroll
        for (int cb = 0; cb < C::kNumBlocks; ++cb)
          tma_load_3d(dst + cb * C::kBlockBytes, str, &full[st], cb * C::kBlockCols, u.h, row);
      }
      ++st_it;
    }
  }
  if (!ok) {
    if (STREAM == 0)
      for (uint32_t i = res_it > C::kNumRes ? res_it - C::kNumRes : 0; i < res_it; ++i)
        mbar_wait_drain(&bars->res_full[i % C::kNumRes], (i / C::kNumRes) & 1);
    for (uint32_t i = st_it > kStages ? st_it - kStages : 0; i < st_it; ++i)
      mbar_wait_drain(&full[i % kStages], (i / kStages) & 1);
  }
}

// ---------------------------------------------------------------- MMA issuer
// Counters of the hand-offs between the MMA issuer and the activation warps.
// Waits on an "empty"/"free" barrier use parity (n & 1) ^ 1 for the n-th use,
// which passes at once on a fresh barrier.
struct XRing {
  uint32_t n = 0;  // X tiles written so far
  template <int NX>
  __device__ __forceinline__ int slot() const { return static_cast<int>(n % NX); }
  template <int NX>
  __device__ __forceinline__ uint32_t full_parity() const { return (n / NX) & 1; }
  template <int NX>
  __device__ __forceinline__ uint32_t empty_parity() const { return ((n / NX) & 1) ^ 1; }
};

// dkdv.  Per query tile i:
//   [P^T(i) in TMEM] dV += P^T(i) dO(i)          (P^T over S^T's columns)
//                    S^T(i+1) = K Q(i+1)^T        (after dV(i) has read P^T)
//   [dS^T(i) in X]   dK += dS^T(i) Q(i)
//   [dP^T(i) loaded] dP^T(i+1) = V dO(i+1)^T
// P^T stays in TMEM (A operand from TMEM) and only dS^T goes through the
// shared X tile, so the two products of a tile never wait on each other for
// X.
// DIRECT (units of segments with dq_direct_segment only): after dK(i),
// dQ(i) = dS(i) K of the unit's only key tile, complete, into kDqCol -- the
// free columns past dK at d <= 64, dP^T's columns at d = 128 (once the
// activation warps have read dP^T(i); dP^T(i+1) then waits until they have
// read dQ(i)).  A separate instantiation, so that the general kernel's code
// is not touched by it.
template <int D>
constexpr uint32_t kDqCol = D <= 64 ? 256 + 2 * D : 128;

template <int D, bool WIN, bool DIRECT>
__device__ void bwd_mma_kv(const BwdParams& p, uint8_t* smem, BwdBars* bars, uint32_t tmem, int n_units,
                           Fail fail) {
  using C = BwdCfg<D, true>;
  const uint32_t res_base = smem_u32(smem + C::kResOff);
  const uint32_t a_base = smem_u32(smem + C::kAOff), b_base = smem_u32(smem + C::kBOff);
  const uint32_t x_base = smem_u32(smem + C::kXOff);
  uint32_t res_it = 0, st_it = 0, acc_it = 0, p_n = 0, dp_n = 0;
  [[maybe_unused]] uint32_t dq_n = 0, dq_w = 0;
  XRing x;
  const bool leader = elect_one();
  bool ok = true;
  // DIRECT: waits until the activation warps have read every dQ issued so far
  [[maybe_unused]] auto dq_read = [&]() -> bool {
    for (; dq_w < dq_n; ++dq_w)
      if (!mbar_wait_warp(&bars->dq_empty, dq_w & 1, fail)) return false;
    return true;
  };
  for (int r = 0; ok; ++r) {
    const int idx = unit_index(r, blockIdx.x, gridDim.x);
    if (idx >= n_units) break;
    const BwdUnit u = bwd_unit<true, WIN>(p, idx);
    if (u.count == 0) continue;
    const int rs = res_it % C::kNumRes;
    if (!(ok = mbar_wait_warp(&bars->res_full[rs], (res_it / C::kNumRes) & 1, fail))) break;
    ++res_it;
    const uint32_t k_t = res_base + rs * C::kResBytes, v_t = k_t + C::kTileBytes;
    {  // S^T and dP^T of the first query tile (S^T after the previous unit's
       // last dV in issue order, which has read its P^T)
      const int sa = st_it % C::kStagesA, sb = st_it % C::kStagesB;
      if (!(ok = mbar_wait_warp(&bars->a_full[sa], (st_it / C::kStagesA) & 1, fail))) break;
      tc_fence_after();
      mma_tile_nt<D>(tmem, k_t, a_base + sa * C::kTileBytes, leader);  // S^T = K Q^T
      if (leader) mma_commit(&bars->s_full);
      if (!(ok = mbar_wait_warp(&bars->dp_free, (dp_n & 1) ^ 1, fail))) break;
      if constexpr (DIRECT && D == 128) {  // (the previous unit's last dQ in dP^T's columns)
        if (!(ok = dq_read())) break;
      }
      if (!(ok = mbar_wait_warp(&bars->b_full[sb], (st_it / C::kStagesB) & 1, fail))) break;
      tc_fence_after();
      mma_tile_nt<D>(tmem + 128, v_t, b_base + sb * C::kTileBytes, leader);  // dP^T = V dO^T
      if (leader) mma_commit(&bars->dp_full);
      ++dp_n;
    }
    for (int i = 0; i < u.count; ++i) {
      const uint32_t it = st_it + i;
      const int sa = it % C::kStagesA, sb = it % C::kStagesB;
      const int sa1 = (it + 1) % C::kStagesA, sb1 = (it + 1) % C::kStagesB;
      const uint32_t q_t = a_base + sa * C::kTileBytes, do_t = b_base + sb * C::kTileBytes;
      const bool more = i + 1 < u.count;
      if (i == 0) {
        if (!(ok = mbar_wait_warp(&bars->acc_empty, (acc_it & 1) ^ 1, fail))) break;
        ++acc_it;
      }
      // dV += P^T dO, P^T in TMEM columns [0,32) (queries 0-63) and [64,96)
      if (!(ok = mbar_wait_warp(&bars->p_full, p_n & 1, fail))) break;
      ++p_n;
      tc_fence_after();
      mma_tile_ts<D>(tmem + 256, tmem, tmem + 64, do_t, i > 0, leader);
      if (leader) mma_commit(&bars->b_empty[sb]);  // dO(i): dP^T(i) and dV(i) issued
      if (more) {  // S^T of the next query tile over the columns dV(i) reads
        if (!(ok = mbar_wait_warp(&bars->a_full[sa1], ((it + 1) / C::kStagesA) & 1, fail))) break;
        tc_fence_after();
        mma_tile_nt<D>(tmem, k_t, a_base + sa1 * C::kTileBytes, leader);
        if (leader) mma_commit(&bars->s_full);
      }
      {  // dK += dS^T Q
        const int xs = x.slot<C::kNumX>();
        if (!(ok = mbar_wait_warp(&bars->x_full[xs], x.full_parity<C::kNumX>(), fail))) break;
        tc_fence_after();
        mma_tile_xs<D>(tmem + 256 + D, x_base + xs * C::kXBytes, q_t, i > 0, leader);
        if constexpr (D <= 64) {
          // fused dQ: this unit's whole contribution dS K (its only query
          // tile), dS read from X as the MN-major A operand and K from the
          // resident tile, into TMEM columns [256 + 2D, 256 + 3D)
          if (p.dq_fused != nullptr) mma_ds_k<D>(tmem + 256 + 2 * D, x_base + xs * C::kXBytes, k_t, leader);
        }
        if constexpr (DIRECT) {  // dQ(i) = dS(i) K, complete: the segment has one key tile
          if constexpr (D == 128) {  // into dP^T's columns, read by now
            if (!(ok = mbar_wait_warp(&bars->dp_free, (dp_n & 1) ^ 1, fail))) break;
          } else {
            if (!(ok = dq_read())) break;
          }
          tc_fence_after();
          mma_ds_k<D>(tmem + kDqCol<D>, x_base + xs * C::kXBytes, k_t, leader);
          if (leader) mma_commit(&bars->dq_full);
          ++dq_n;
        }
        if (leader) mma_commit(&bars->x_empty[xs]);
        if (leader) mma_commit(&bars->a_empty[sa]);  // Q(i): S^T(i) and dK(i) issued
        ++x.n;
      }
      if (more) {  // dP^T of the next query tile, once dP^T(i) (DIRECT, d = 128: and dQ(i)) is read
        if (!(ok = mbar_wait_warp(&bars->dp_free, (dp_n & 1) ^ 1, fail))) break;
        if constexpr (DIRECT && D == 128) {
          if (!(ok = dq_read())) break;
        }
        if (!(ok = mbar_wait_warp(&bars->b_full[sb1], ((it + 1) / C::kStagesB) & 1, fail))) break;
        tc_fence_after();
        mma_tile_nt<D>(tmem + 128, v_t, b_base + sb1 * C::kTileBytes, leader);
        if (leader) mma_commit(&bars->dp_full);
        ++dp_n;
      }
    }
    if (!ok) break;
    st_it += u.count;
    if (leader) mma_commit(&bars->acc_full);
    if (leader) mma_commit(&bars->res_empty[rs]);
  }
  if (leader) mma_commit(&bars->drain);
  mbar_wait_drain(&bars->drain, 0);
}

// dq.  Per key tile i:
//   [S(i) loaded]  S(i+1) = Q K(i+1)^T
//   [dS(i) in X]   dQ += dS(i) K(i)
//   [dP(i) loaded] dP(i+1) = dO V(i+1)^T
// dP(i+1) goes last because with a single V stage its operand can only land
// after dP(i) has completed.
template <int D, bool WIN>
__device__ void bwd_mma_q(const BwdParams& p, uint8_t* smem, BwdBars* bars, uint32_t tmem, int n_units,
                          Fail fail) {
  using C = BwdCfg<D, false>;
  const uint32_t res_base = smem_u32(smem + C::kResOff);
  const uint32_t a_base = smem_u32(smem + C::kAOff), b_base = smem_u32(smem + C::kBOff);
  const uint32_t x_base = smem_u32(smem + C::kXOff);
  uint32_t res_it = 0, st_it = 0, acc_it = 0, s_n = 0, dp_n = 0;
  XRing x;
  const bool leader = elect_one();
  bool ok = true;
  for (int r = 0; ok; ++r) {
    const int idx = unit_index(r, blockIdx.x, gridDim.x);
    if (idx >= n_units) break;
    const BwdUnit u = bwd_unit<false, WIN>(p, idx);
    if (u.count == 0) continue;
    const int rs = res_it % C::kNumRes;
    if (!(ok = mbar_wait_warp(&bars->res_full[rs], (res_it / C::kNumRes) & 1, fail))) break;
    ++res_it;
    const uint32_t q_t = res_base + rs * C::kResBytes, do_t = q_t + C::kTileBytes;
    {  // S and dP of the first key tile
      const int sa = st_it % C::kStagesA, sb = st_it % C::kStagesB;
      if (!(ok = mbar_wait_warp(&bars->s_free, (s_n & 1) ^ 1, fail))) break;
      if (!(ok = mbar_wait_warp(&bars->a_full[sa], (st_it / C::kStagesA) & 1, fail))) break;
      tc_fence_after();
      mma_tile_nt<D>(tmem, q_t, a_base + sa * C::kTileBytes, leader);  // S = Q K^T
      if (leader) mma_commit(&bars->s_full);
      ++s_n;
      if (!(ok = mbar_wait_warp(&bars->dp_free, (dp_n & 1) ^ 1, fail))) break;
      if (!(ok = mbar_wait_warp(&bars->b_full[sb], (st_it / C::kStagesB) & 1, fail))) break;
      tc_fence_after();
      mma_tile_nt<D>(tmem + 128, do_t, b_base + sb * C::kTileBytes, leader);  // dP = dO V^T
      if (leader) mma_commit(&bars->dp_full);
      if (leader) mma_commit(&bars->b_empty[sb]);  // V is read by dP only
      ++dp_n;
    }
    for (int i = 0; i < u.count; ++i) {
      const uint32_t it = st_it + i;
      const int sa = it % C::kStagesA;
      const int sa1 = (it + 1) % C::kStagesA, sb1 = (it + 1) % C::kStagesB;
      const uint32_t k_t = a_base + sa * C::kTileBytes;
      const bool more = i + 1 < u.count;
      if (more) {
        if (!(ok = mbar_wait_warp(&bars->s_free, (s_n & 1) ^ 1, fail))) break;
        if (!(ok = mbar_wait_warp(&bars->a_full[sa1], ((it + 1) / C::kStagesA) & 1, fail))) break;
        tc_fence_after();
        mma_tile_nt<D>(tmem, q_t, a_base + sa1 * C::kTileBytes, leader);
        if (leader) mma_commit(&bars->s_full);
        ++s_n;
      }
      if (i == 0) {
        if (!(ok = mbar_wait_warp(&bars->acc_empty, (acc_it & 1) ^ 1, fail))) break;
        ++acc_it;
      }
      const int xs = x.slot<C::kNumX>();
      if (!(ok = mbar_wait_warp(&bars->x_full[xs], x.full_parity<C::kNumX>(), fail))) break;
      tc_fence_after();
      mma_tile_xs<D>(tmem + 256, x_base + xs * C::kXBytes, k_t, i > 0, leader);  // dQ += dS K
      if (leader) mma_commit(&bars->x_empty[xs]);
      if (leader) mma_commit(&bars->a_empty[sa]);  // K(i): S(i) and dQ(i) issued
      ++x.n;
      if (more) {
        if (!(ok = mbar_wait_warp(&bars->dp_free, (dp_n & 1) ^ 1, fail))) break;
        if (!(ok = mbar_wait_warp(&bars->b_full[sb1], ((it + 1) / C::kStagesB) & 1, fail))) break;
        tc_fence_after();
        mma_tile_nt<D>(tmem + 128, do_t, b_base + sb1 * C::kTileBytes, leader);
        if (leader) mma_commit(&bars->dp_full);
        if (leader) mma_commit(&bars->b_empty[sb1]);
        ++dp_n;
      }
    }
    if (!ok) break;
    st_it += u.count;
    if (leader) mma_commit(&bars->acc_full);
    if (leader) mma_commit(&bars->res_empty[rs]);
  }
  if (leader) mma_commit(&bars->drain);
  mbar_wait_drain(&bars->drain, 0);
}

// ----------------------------------------------------------- dS store role
// dK/dV pass with stored dS: every dS^T tile the activation warps put in X is
// also copied to the scratch array by TMA (one elected lane of warp 3); the X
// slot is released once both the dK MMA and this copy have read it.
template <int D, bool WIN>
__device__ void bwd_ds_store(const BwdParams& p, uint8_t* smem, BwdBars* bars, int n_units, Fail fail) {
  using C = BwdCfg<D, true>;
  uint8_t* x_base = smem + C::kXOff;
  XRing x;
  const bool leader = elect_one();
  const uint64_t policy = l2_evict_first_policy();
  bool ok = true;
  for (int r = 0; ok; ++r) {
    const int idx = unit_index(r, blockIdx.x, gridDim.x);
    if (idx >= n_units) break;
    const BwdUnit u = bwd_unit<true, WIN>(p, idx);
    if (u.count == 0) continue;
    // a segment whose dS tiles do not fit the scratch gets its dQ by
    // recomputation: nothing is stored, the X tiles are only released
    const bool store = __ldg(p.ds_base + u.b) >= 0;
    for (int i = 0; i < u.count; ++i) {
      const int xs = x.slot<C::kNumX>();
      if (!(ok = mbar_wait_warp(&bars->x_full[xs], x.full_parity<C::kNumX>(), fail))) break;
      if (leader && !store) mbar_arrive(&bars->x_empty[xs]);
      if (leader && store) {
        const int row = ds_row(p.ds_base, u.seg, u.b, u.h, u.tile, u.first + i, WIN ? p.window : 0);
        const uint8_t* src = x_base + xs * C::kXBytes;
        tma_store_2d_hint(&p.tm_ds, src, 0, row, policy);
        // at d <= 64, the upper 64 query columns only where a query row of
        // the segment reaches them (the dQ pass never reads them otherwise;
        // at d = 128 the branch measured slower in this pass)
        if (D == 128 || u.seg.lq - (u.first + i) * kTile > kTile / 2)
          tma_store_2d_hint(&p.tm_ds, src + C::kXBytes / 2, kTile / 2, row, policy);
        bulk_commit();
        bulk_wait_read_all();
        mbar_arrive(&bars->x_empty[xs]);
      }
      __syncwarp();
      ++x.n;
    }
  }
  if (leader) bulk_wait_all();
  __syncwarp();
}

// Fused dQ: row r (a shared query row) of the dQ contribution block of unit
// (segment b, head h, key tile kt), [q_rows][D] fp32 per block.
template <int D>
__device__ __forceinline__ float* dq_fused_row(const BwdParams& p, const BwdUnit& u, int r) {
  const int64_t block = (static_cast<int64_t>(__ldg(p.kv_item_base + u.b)) + u.tile) * p.heads + u.h;
  return p.dq_fused + (block * p.q_rows + r) * D;
}

// --------------------------------------------------------- activation warps
// Geometry of one (own tile, partner tile) pair for the thread of row r.
// KV-major: own row = key j, column c = query i; Q-major: own row = query i,
// column c = key j.  rel = i - j = rel0 + sgn * c.  Valid columns are
// lo <= c < hi (the subtraction scheme: both bounds computed once per tile).
struct PairGeom {
  int lo, hi;
  int rel0, sgn;
  bool masked;   // some column of some row of this warp is invalid
  bool band;     // some |rel| < R in this tile (per-element bias)
  bool upper;    // not band: every rel >= R (else every rel <= -R)
  float bconst;  // the bias of every element when not band (0 without a table)
};

// bc_lo / bc_hi: the table's two end entries (the bias of every element of
// a tile that lies wholly below -R / above +R), loaded once per unit.
template <bool KV_MAJOR, bool WIN>
__device__ __forceinline__ PairGeom pair_geom(const BwdParams& p, const BwdUnit& u, int pt, int r, bool row_ok,
                                              const float* brow, int R, float bc_lo, float bc_hi) {
  PairGeom g;
  g.lo = 0;
  if constexpr (KV_MAJOR) {
    g.hi = min(kTile, u.seg.lq - pt * kTile);
    if (p.causal && pt == u.tile) g.lo = r;               // i >= j  <=>  c >= r
    g.rel0 = (pt - u.tile) * kTile - r;
    g.sgn = 1;
  } else {
    g.hi = min(kTile, u.seg.lkv - pt * kTile);
    if (p.causal && pt == u.tile) g.hi = min(g.hi, r + 1);  // j <= i  <=>  c <= r
    g.rel0 = (u.tile - pt) * kTile + r;
    g.sgn = -1;
  }
  if constexpr (WIN) {  // |rel| < w with rel = rel0 + sgn c; each bound is formed only where it binds
    const int w = p.window;
    if (KV_MAJOR) {
      if (g.rel0 <= -w) g.lo = max(g.lo, 1 - w - g.rel0);
      if (g.rel0 > w - kTile) g.hi = min(g.hi, w - g.rel0);
    } else {
      if (g.rel0 >= w) g.lo = max(g.lo, g.rel0 - w + 1);
      if (g.rel0 < kTile - w) g.hi = min(g.hi, g.rel0 + w);
    }
  }
  if (!row_ok) g.hi = 0;
  g.masked = __any_sync(0xffffffffu, g.lo > 0 || g.hi < kTile);
  const int relmin = (KV_MAJOR ? (pt - u.tile) : (u.tile - pt)) * kTile - (kTile - 1);
  const int relmax = relmin + 2 * (kTile - 1);
  g.band = brow != nullptr && relmin < R && relmax > -R;
  g.upper = relmin >= R;
  g.bconst = g.upper ? bc_hi : bc_lo;
  return g;
}

__device__ __forceinline__ float bias_lookup(const float* brow, int rel, int R) {
  return ld_nc_f32(brow + min(max(rel, -R), R) + R);
}

// Phase A on one 32-column chunk: x from S (+ bias), P (bf16, packed into pk)
// and what phase B needs (act'(x), or P for softmax) into keep.  BAND and
// MASKED are decided once per tile; CHUNK (0 or 1) selects which of the
// thread's 16-column groups take the ALU route (GELU/SiLU).
template <int ACT, bool KV_MAJOR, int CHUNK, bool BAND, bool MASKED>
__device__ __forceinline__ void phase_a_chunk(const uint32_t (&sv)[32], const float (&lse_c)[32], float lse2_row,
                                              const PairGeom& g, const float* brow, int R, int cbase, float hs,
                                              float s2, float (&keep)[32], uint32_t (&pk)[16]) {
  constexpr bool kSoftmax = ACT == 2;
  const float hb = 0.5f * g.bconst;
  const float b2 = kLog2e * g.bconst;
#pragma unroll
  for (int e2 = 0; e2 < 16; ++e2) {
    const int cl = 2 * e2, c = cbase + cl;
    const float2 sval = make_float2(__uint_as_float(sv[cl]), __uint_as_float(sv[cl + 1]));
    float2 bias = f2(g.bconst);
    if constexpr (BAND)
      bias = make_float2(bias_lookup(brow, g.rel0 + g.sgn * c, R), bias_lookup(brow, g.rel0 + g.sgn * (c + 1), R));
    float2 pv, kv;
    if constexpr (kSoftmax) {
      const float2 x2 = BAND ? __ffma2_rn(sval, f2(s2), __fmul2_rn(bias, f2(kLog2e))) : __ffma2_rn(sval, f2(s2), f2(b2));
      const float2 l2 = KV_MAJOR ? make_float2(lse_c[cl], lse_c[cl + 1]) : f2(lse2_row);
      const float2 z = __fadd2_rn(x2, make_float2(-l2.x, -l2.y));
      pv = make_float2(ex2_sfu(z.x), ex2_sfu(z.y));
      kv = pv;
    } else {
      const float2 hx = BAND ? __ffma2_rn(sval, f2(hs), __fmul2_rn(bias, f2(0.5f))) : __ffma2_rn(sval, f2(hs), f2(hb));
      // the last kBwdAluGroups of the four 16-column groups take the ALU route
      if (CHUNK * 2 + (e2 >= 8 ? 1 : 0) >= 4 - kBwdAluGroups) pv = act2_d<ACT, true>(hx, kv);
      else pv = act2_d<ACT, false>(hx, kv);
    }
    if constexpr (MASKED) {
      if (!(c >= g.lo && c < g.hi)) {
        pv.x = 0.f;
        kv.x = 0.f;
      }
      if (!(c + 1 >= g.lo && c + 1 < g.hi)) {
        pv.y = 0.f;
        kv.y = 0.f;
      }
    }
    keep[cl] = kv.x;
    keep[cl + 1] = kv.y;
    pk[e2] = pack_bf16(pv.x, pv.y);
  }
}

// Phase B on one 32-column chunk: dS = act'(x) dP (softmax: P (dP - D)),
// packed into pk.  DBIAS: 0 none, 1 the tile clamps to one table end (sum
// into row_sum), 2 per-element table entries (band tile).
//
// Band tiles (KV-major): element (lane l, chunk column m) of a warp has
// rel = W + m - l with W uniform over the warp and chunk, so it belongs to
// diagonal d = m - l in [-31, 31].  At column m lane L takes the value of
// lane (m - L) mod 32 by a shuffle, whose diagonal is L if m >= L and L - 32
// otherwise; each lane thus sums two diagonals per chunk.  Chunk 1's W is
// chunk 0's plus 32, so its lower diagonal is chunk 0's upper one, and the
// three sums dacc[0..2] hold the diagonals W0 + L - 32, W0 + L, W0 + L + 32.
template <int ACT, bool KV_MAJOR, int DBIAS, int CHUNK>
__device__ __forceinline__ void phase_b_chunk(const uint32_t (&dv)[32], const float (&del_c)[32], float delta_row,
                                              const float (&keep)[32], float2& row_sum, float (&dacc)[3],
                                              uint32_t (&pk)[16]) {
  constexpr bool kSoftmax = ACT == 2;
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int e2 = 0; e2 < 16; ++e2) {
    const int cl = 2 * e2;
    const float2 dp = make_float2(__uint_as_float(dv[cl]), __uint_as_float(dv[cl + 1]));
    const float2 kv = make_float2(keep[cl], keep[cl + 1]);
    float2 ds;
    if constexpr (kSoftmax) {
      const float2 dl = KV_MAJOR ? make_float2(del_c[cl], del_c[cl + 1]) : f2(delta_row);
      ds = __fmul2_rn(kv, __fadd2_rn(dp, make_float2(-dl.x, -dl.y)));
    } else {
      ds = __fmul2_rn(dp, kv);
    }
    pk[e2] = pack_bf16(ds.x, ds.y);
    if constexpr (DBIAS == 1) row_sum = __fadd2_rn(row_sum, ds);
    if constexpr (DBIAS == 2) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int m = cl + e;
        const float v = __shfl_sync(0xffffffffu, e ? ds.y : ds.x, (m - lane) & 31);
        if (m >= lane) dacc[CHUNK + 1] += v;
        else dacc[CHUNK] += v;
      }
    }
  }
}

// DIRECT: dQ of query tile qt (key-major pass): TMEM lane r is query row r
// of the tile; warpgroup `half` owns columns [half D/2, (half+1) D/2).
// Scaled by s into dq (bf16), or into dq_part (fp32) with shared queries.
// At d = 128 into dq the warp stages its 32 rows x 64 columns in its own 4 KB
// of the X tile (free here: dK and this dQ have read it, and phase B writes
// it only after this), which leaves by one TMA store when the 32 rows lie in
// the segment and by stores of four whole 128-byte rows per instruction
// otherwise: a thread's own row pieces lie H D 2 bytes apart, and storing
// them directly touched 32 lines per instruction (~2 K cycles of the
// load/store unit per tile in the traces).
template <int D>
__device__ __forceinline__ bool read_dq(const BwdParams& p, BwdBars* bars, uint32_t t_dq, int half, int r, int q0,
                                        int lq, int h, int qt, uint32_t parity, Fail fail, uint8_t* stage) {
  if (!mbar_wait(&bars->dq_full, parity, fail)) return false;
  tc_fence_after();
  if constexpr (D == 128) {
    if (p.dq_part == nullptr) {
      const int lr = threadIdx.x & 31, quad = r >> 5;
      const uint32_t stg = smem_u32(stage);
      if (lr == 0) bulk_wait_read_all();  // this warp's previous TMA store has read the block
      __syncwarp();
#pragma unroll
      for (int c0 = 0; c0 < 64; c0 += 32) {
        uint32_t o[32];
        tmem_ld32(t_dq + c0, o);
        tmem_ld_wait(o);
        if (c0 == 32) {  // every column of this tile's dQ is in registers
          tc_fence_before();
          mbar_arrive_warp(&bars->dq_empty);
        }
#pragma unroll
        for (int c = 0; c < 32; c += 8) {
          uint32_t w[4];
#pragma unroll
          for (int e = 0; e < 4; ++e)
            w[e] = pack_bf16(__uint_as_float(o[c + 2 * e]) * p.scale, __uint_as_float(o[c + 2 * e + 1]) * p.scale);
          const int j = (c0 + c) >> 3;
          st_shared_v4(stg + lr * 128 + ((j ^ (lr & 7)) << 4), w[0], w[1], w[2], w[3]);
        }
      }
      const int rows = lq - qt * kTile;
      const int row0 = q0 + qt * kTile + quad * 32;  // the warp's first row
      if (quad * 32 + 31 < rows) {
        fence_proxy_async_smem();
        __syncwarp();
        if (lr == 0) {
          tma_store_3d(&p.tm_dq, stage, 64 * half, h, row0);
          bulk_commit();
        }
      } else {
        __syncwarp();
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int rw = 4 * k + (lr >> 3), j = lr & 7;
          uint32_t a, b2, c2, d2;
          ld_shared_v4(stg + rw * 128 + ((j ^ (rw & 7)) << 4), a, b2, c2, d2);
          if (quad * 32 + rw < rows)
            st_global_v4(p.dq + ((static_cast<int64_t>(row0) + rw) * p.heads + h) * D + 64 * half + 8 * j, a, b2,
                         c2, d2);
        }
        __syncwarp();
      }
      return true;
    }
  }
  const bool q_ok = qt * kTile + r < lq;
  const int64_t qrow = (static_cast<int64_t>(q0) + qt * kTile + r) * p.heads + h;
  constexpr int kChunk = D / 2 < 32 ? D / 2 : 32;
#pragma unroll
  for (int c0 = 0; c0 < D / 2; c0 += kChunk) {
    uint32_t o[32];
    if constexpr (kChunk == 32) {
      tmem_ld32(t_dq + c0, o);
      tmem_ld_wait(o);
    } else {
      uint32_t(&o16)[16] = *reinterpret_cast<uint32_t(*)[16]>(o);
      tmem_ld16(t_dq + c0, o16);
      tmem_ld_wait16(o16);
    }
    if (c0 + kChunk == D / 2) {  // every column of this tile's dQ is in registers
      tc_fence_before();
      mbar_arrive_warp(&bars->dq_empty);
    }
    if (q_ok) {
      const int col = (D / 2) * half + c0;
      if (p.dq_part) {
#pragma unroll
        for (int c = 0; c < kChunk; c += 4)
          st_global_v4(p.dq_part + qrow * D + col + c, __float_as_uint(__uint_as_float(o[c]) * p.scale),
                       __float_as_uint(__uint_as_float(o[c + 1]) * p.scale),
                       __float_as_uint(__uint_as_float(o[c + 2]) * p.scale),
                       __float_as_uint(__uint_as_float(o[c + 3]) * p.scale));
      } else {
#pragma unroll
        for (int c = 0; c < kChunk; c += 8) {
          uint32_t w[4];
#pragma unroll
          for (int e = 0; e < 4; ++e)
            w[e] = pack_bf16(__uint_as_float(o[c + 2 * e]) * p.scale, __uint_as_float(o[c + 2 * e + 1]) * p.scale);
          st_global_v4(p.dq + qrow * D + col + c, w[0], w[1], w[2], w[3]);
        }
      }
    }
  }
  return true;
}

template <int D, int ACT, bool KV_MAJOR, bool WIN, bool DIRECT>
__device__ void bwd_act(const BwdParams& p, uint8_t* smem, BwdBars* bars, uint32_t tmem, int n_units, Fail fail) {
  using C = BwdCfg<D, KV_MAJOR>;
  constexpr bool kSoftmax = ACT == 2;
  const int warp = threadIdx.x >> 5;
  const int quad = warp & 3;
  const int half = (warp - 4) >> 2;                // which 64 columns this warpgroup owns
  const int r = quad * 32 + (threadIdx.x & 31);    // row of this unit's own tile
  const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
  const uint32_t t_s = tmem + lane_off + 64 * half;
  const uint32_t t_dp = tmem + lane_off + 128 + 64 * half;
  const uint32_t x_base = smem_u32(smem + C::kXOff);
  const int H = p.heads;
  const bool want_dbias = KV_MAJOR && p.dbias_part != nullptr;
  const int R = (p.bias_len - 1) / 2;
  uint32_t s_it = 0, dp_it = 0, acc_it = 0;
  [[maybe_unused]] uint32_t dq_it = 0;
  // DIRECT at d = 128: this warp's 4 KB of the X tile (its rows, its
  // warpgroup's column block) stages dQ for its TMA store
  [[maybe_unused]] uint8_t* dq_stage = smem + C::kXOff + half * (kTile * 128) + quad * 32 * 128;
  [[maybe_unused]] const uint32_t t_dq = tmem + lane_off + kDqCol<D> + (D / 2) * half;  // DIRECT: dQ columns
  XRing x;
  const float hs = 0.5f * p.scale;                 // x / 2 = hs S + bias / 2
  const float s2 = p.scale * kLog2e;               // softmax: x log2 e

  for (int rr = 0;; ++rr) {
    const int idx = unit_index(rr, blockIdx.x, gridDim.x);
    if (idx >= n_units) break;
    const BwdUnit u = bwd_unit<KV_MAJOR, WIN>(p, idx);
    if (u.rows <= 0) continue;
    const bool row_ok = r < u.rows;
    const int64_t grow = static_cast<int64_t>(KV_MAJOR ? u.seg.k0 : u.seg.q0) + u.tile * kTile + r;
    const float* brow = p.bias_len ? p.bias + static_cast<int64_t>(u.h) * p.bias_len : nullptr;
    unsigned long long* part =
        want_dbias ? p.dbias_part + (static_cast<int64_t>(blockIdx.x) * H + u.h) * p.bias_len : nullptr;
    float acc_lo = 0.f, acc_hi = 0.f;  // dbias mass clamped to the table's ends
    const float bc_lo = brow ? __ldg(brow) : 0.f, bc_hi = brow ? __ldg(brow + 2 * R) : 0.f;

    if (u.count == 0) {  // no partner rows: the gradient rows are zero
      if constexpr (KV_MAJOR && D <= 64) {
        if (p.dq_fused != nullptr && r < p.q_rows) {  // (so is this unit's dQ contribution)
          float* dst = dq_fused_row<D>(p, u, r) + half * (D / 2);
#pragma unroll
          for (int c = 0; c < D / 2; c += 4) st_global_v4(dst + c, 0u, 0u, 0u, 0u);
        }
      }
      if (row_ok) {
        if constexpr (KV_MAJOR) {
          __nv_bfloat16* dst = (half == 0 ? p.dv : p.dk) + (grow * H + u.h) * D;
#pragma unroll
          for (int c = 0; c < D; c += 8) st_global_v4(dst + c, 0u, 0u, 0u, 0u);
        } else if (p.dq_part) {
          float* dst = p.dq_part + (grow * H + u.h) * D + half * (D / 2);
#pragma unroll
          for (int c = 0; c < D / 2; c += 4) st_global_v4(dst + c, 0u, 0u, 0u, 0u);
        } else {
          __nv_bfloat16* dst = p.dq + (grow * H + u.h) * D + half * (D / 2);
#pragma unroll
          for (int c = 0; c < D / 2; c += 8) st_global_v4(dst + c, 0u, 0u, 0u, 0u);
        }
      }
      continue;
    }

    // softmax: per-row statistics of the query rows this thread owns (dq)
    float lse2_row = 0.f, delta_row = 0.f;
    if constexpr (kSoftmax && !KV_MAJOR) {
      if (row_ok) {
        lse2_row = p.lse[static_cast<int64_t>(u.h) * p.total_q + grow] * kLog2e;
        delta_row = p.delta[static_cast<int64_t>(u.h) * p.total_q + grow];
      }
    }

    bool ok = true;
    for (int i = 0; i < u.count; ++i) {
      const int pt = u.first + i;  // partner tile
      const PairGeom g = pair_geom<KV_MAJOR, WIN>(p, u, pt, r, row_ok, brow, R, bc_lo, bc_hi);
      // softmax, key-major: log2-scaled LSE and D of the query columns this
      // warpgroup owns, one value per lane and 32-column chunk, loaded before
      // the wait for S and broadcast by shuffles (every query tile is new to
      // L1: loads issued at their use would wait on L2 four times per tile)
      float cur_lse[2] = {0.f, 0.f}, cur_del[2] = {0.f, 0.f};
      if constexpr (kSoftmax && KV_MAJOR) {
        const int c0 = 64 * half + (threadIdx.x & 31);
        const int64_t q0 = static_cast<int64_t>(u.h) * p.total_q + u.seg.q0 + pt * kTile + c0;
        const int lim = u.seg.lq - pt * kTile - c0;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          cur_lse[c] = 32 * c < lim ? __ldg(p.lse + q0 + 32 * c) * kLog2e : 0.f;
          cur_del[c] = 32 * c < lim ? __ldg(p.delta + q0 + 32 * c) : 0.f;
        }
      }

      // ---- S (S^T) of this tile into registers; its TMEM columns go back to
      // the MMA issuer for the next tile
      if (!(ok = mbar_wait(&bars->s_full, s_it & 1, fail))) break;
      ++s_it;
      tc_fence_after();
      // 32-column chunks of this warpgroup's 64 columns that hold a partner
      // row of the segment (the same for every thread); phase B skips the
      // others and writes zero dS there; phase A skips them at d <= 64 and
      // otherwise zeroes their P through its mask
      const int ncols = (KV_MAJOR ? u.seg.lq : u.seg.lkv) - pt * kTile - 64 * half;
      const int live = ncols >= 33 ? 2 : (ncols >= 1 ? 1 : 0);
      uint32_t sv0[32], sv1[32];
      tmem_ld32(t_s, sv0);
      tmem_ld32(t_s + 32, sv1);
      tmem_ld_wait2(sv0, sv1);
      if constexpr (!KV_MAJOR) {  // dkdv reuses these columns for P^T instead
        tc_fence_before();
        mbar_arrive_warp(&bars->s_free);
      }

      // ---- phase A: S -> (P, act'(x)) [softmax: P]; P^T to X (dkdv)
      float keep0[32], keep1[32];  // act'(x) (GELU/SiLU) or P (softmax) per owned column
#pragma unroll
      for (int chunk = 0; chunk < 2; ++chunk) {
        if constexpr (DIRECT && D == 128) {
          // the previous query tile's dQ, between the two halves of phase A:
          // it is complete by then, and this tile's dP^T (into the same
          // columns) then runs during the second half
          if (chunk == 1 && i > 0) {
            if (!(ok = read_dq<D>(p, bars, t_dq, half, r, u.seg.q0, u.seg.lq, u.h, pt - 1, dq_it & 1, fail,
                                  dq_stage)))
              break;
            ++dq_it;
          }
        }
        if constexpr (D <= 64) {  // (at d = 128 this branch makes ptxas spill in the hot loop)
          if (chunk >= live) {    // no partner row in these columns: P^T (and later dS) zero
            if constexpr (KV_MAJOR) {
              const uint32_t zero[16] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
              tmem_st16(t_s + 16 * chunk, zero);
            }
            continue;
          }
        }
        const int cbase = 64 * half + 32 * chunk;
        const uint32_t(&sv)[32] = chunk == 0 ? sv0 : sv1;
        uint32_t pk[16];
        float(&keep)[32] = chunk == 0 ? keep0 : keep1;
        float lse_c[32];
        if constexpr (kSoftmax && KV_MAJOR) {
#pragma unroll
          for (int e = 0; e < 32; ++e) lse_c[e] = __shfl_sync(0xffffffffu, cur_lse[chunk], e);
        }
#define JG_PHASE_A(CH, BAND, MASKED)                                                                         \
  phase_a_chunk<ACT, KV_MAJOR, CH, BAND, MASKED>(sv, lse_c, lse2_row, g, brow, R, cbase, hs, s2, keep, pk)
        if (chunk == 0) {
          if (g.band) {
            if (g.masked) JG_PHASE_A(0, true, true); else JG_PHASE_A(0, true, false);
          } else {
            if (g.masked) JG_PHASE_A(0, false, true); else JG_PHASE_A(0, false, false);
          }
        } else {
          if (g.band) {
            if (g.masked) JG_PHASE_A(1, true, true); else JG_PHASE_A(1, true, false);
          } else {
            if (g.masked) JG_PHASE_A(1, false, true); else JG_PHASE_A(1, false, false);
          }
        }
#undef JG_PHASE_A
        if constexpr (KV_MAJOR) tmem_st16(t_s + 16 * chunk, pk);  // P^T over S^T columns already read
      }
      if (!ok) break;
      if constexpr (KV_MAJOR) {
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive_warp(&bars->p_full);
      }
      if constexpr (DIRECT && D <= 64) {  // the previous query tile's dQ (its own columns)
        if (i > 0) {
          if (!(ok = read_dq<D>(p, bars, t_dq, half, r, u.seg.q0, u.seg.lq, u.h, pt - 1, dq_it & 1, fail,
                                dq_stage)))
            break;
          ++dq_it;
        }
      }

      // ---- phase B: dP -> dS (bf16 into X), dbias partial sums
      if (!(ok = mbar_wait(&bars->dp_full, dp_it & 1, fail))) break;
      ++dp_it;
      tc_fence_after();
      float2 row_sum = f2(0.f);
      float dacc[3] = {0.f, 0.f, 0.f};
      const int dmode = !want_dbias ? 0 : (g.band ? 2 : 1);
      // dP columns are loaded one 32-column chunk at a time (both halves of
      // dP and of act' live at once would exceed the register budget); the
      // TMEM columns go back after the second load -- the next dP is not
      // needed before the next tile's phase B.
#pragma unroll
      for (int chunk = 0; chunk < 2; ++chunk) {
        uint32_t dv[32];
        tmem_ld32(t_dp + 32 * chunk, dv);
        tmem_ld_wait(dv);
        if (chunk == 1) {
          tc_fence_before();
          mbar_arrive_warp(&bars->dp_free);
        }
        uint32_t pk[16];
        if (chunk < live) {
          float del_c[32];
          if constexpr (kSoftmax && KV_MAJOR) {
#pragma unroll
            for (int e = 0; e < 32; ++e) del_c[e] = __shfl_sync(0xffffffffu, cur_del[chunk], e);
          }
          const float(&keep)[32] = chunk == 0 ? keep0 : keep1;
#define JG_PHASE_B(DB) \
  phase_b_chunk<ACT, KV_MAJOR, DB, 0>(dv, del_c, delta_row, keep, row_sum, dacc, pk)
#define JG_PHASE_B1(DB) \
  phase_b_chunk<ACT, KV_MAJOR, DB, 1>(dv, del_c, delta_row, keep, row_sum, dacc, pk)
          if (chunk == 0) {
            if (dmode == 0) JG_PHASE_B(0); else if (dmode == 1) JG_PHASE_B(1); else JG_PHASE_B(2);
          } else {
            if (dmode == 0) JG_PHASE_B1(0); else if (dmode == 1) JG_PHASE_B1(1); else JG_PHASE_B1(2);
          }
#undef JG_PHASE_B
#undef JG_PHASE_B1
        } else {
#pragma unroll
          for (int e = 0; e < 16; ++e) pk[e] = 0u;
        }
        if (chunk == 0 && !(ok = mbar_wait(&bars->x_empty[x.slot<C::kNumX>()], x.empty_parity<C::kNumX>(), fail)))
          break;
        if constexpr (DIRECT && D == 128) {  // the dQ staged in X has been read by its TMA store
          if (chunk == 0) {
            if ((threadIdx.x & 31) == 0) bulk_wait_read_all();
            __syncwarp();
          }
        }
        store_x_chunk(x_base + x.slot<C::kNumX>() * C::kXBytes, half, chunk, r, pk);
      }
      if (!ok) break;
      fence_proxy_async_smem();
      mbar_arrive_warp(&bars->x_full[x.slot<C::kNumX>()]);
      ++x.n;
      if (dmode == 1) {
        if (g.upper) acc_hi += row_sum.x + row_sum.y;  // the whole tile clamps to one end of the table
        else acc_lo += row_sum.x + row_sum.y;
      } else if (dmode == 2) {
        // diagonal sums -> table entries (rel of diagonal k: see phase_b_chunk)
        const int rel1 = g.rel0 + 2 * (threadIdx.x & 31) + 64 * half;
#pragma unroll
        for (int k = 0; k < 3; ++k) {
          const int rel = rel1 + 32 * (k - 1);
          if (rel >= R) acc_hi += dacc[k];
          else if (rel <= -R) acc_lo += dacc[k];
          else atomicAdd(part + rel + R, dbias_fixed(dacc[k]));
        }
      }
    }
    if (!ok) break;
    if constexpr (DIRECT) {
      if (!read_dq<D>(p, bars, t_dq, half, r, u.seg.q0, u.seg.lq, u.h, u.first + u.count - 1, dq_it & 1, fail,
                      dq_stage))
        break;
      ++dq_it;
    }

    // epilogue
    if (!mbar_wait(&bars->acc_full, acc_it & 1, fail)) break;
    ++acc_it;
    tc_fence_after();
    if constexpr (KV_MAJOR && D >= 64) {
      // warpgroup 0 stores dV, warpgroup 1 stores dK (scaled by s).  A thread
      // owns one row and rows lie H D 2 bytes apart, so plain stores would
      // touch 32 lines per instruction.  The warp stages 64 columns of its 32
      // rows at a time in its own 4 KB block of the next X slot (the rows and
      // columns it writes dS to in phase B, free once that slot is empty),
      // then stores four whole 128-byte row pieces per instruction.
      const uint32_t t_acc = tmem + lane_off + 256 + D * half;
      const float mul = half == 0 ? 1.0f : p.scale;
      const int xs = x.slot<C::kNumX>();
      if (!mbar_wait(&bars->x_empty[xs], x.empty_parity<C::kNumX>(), fail)) break;
      const int lr = threadIdx.x & 31;
      if constexpr (DIRECT && D == 128) {  // the dQ staged in X has been read by its TMA store
        if (lr == 0) bulk_wait_read_all();
        __syncwarp();
      }
      const uint32_t blk = x_base + xs * C::kXBytes + half * (kTile * 128) + quad * 32 * 128;
      __nv_bfloat16* base = half == 0 ? p.dv : p.dk;
      const int64_t row0 = grow - lr;  // global row of the warp's first row
#pragma unroll
      for (int hb = 0; hb < D / 64; ++hb) {
#pragma unroll
        for (int c0 = 0; c0 < 64; c0 += 32) {
          uint32_t o[32];
          tmem_ld32(t_acc + 64 * hb + c0, o);
          tmem_ld_wait(o);
#pragma unroll
          for (int c = 0; c < 32; c += 8) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
              w[e] = pack_bf16(__uint_as_float(o[c + 2 * e]) * mul, __uint_as_float(o[c + 2 * e + 1]) * mul);
            const int j = (c0 + c) >> 3;  // 16-byte chunk of the 128-byte piece
            st_shared_v4(blk + lr * 128 + ((j ^ (lr & 7)) << 4), w[0], w[1], w[2], w[3]);
          }
        }
        __syncwarp();
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int rr = 4 * k + (lr >> 3), j = lr & 7;
          uint32_t a, b2, c2, d2;
          ld_shared_v4(blk + rr * 128 + ((j ^ (rr & 7)) << 4), a, b2, c2, d2);
          if (quad * 32 + rr < u.rows)
            st_global_v4(base + ((row0 + rr) * H + u.h) * D + 64 * hb + 8 * j, a, b2, c2, d2);
        }
        __syncwarp();
      }
    } else if constexpr (KV_MAJOR) {
      // warpgroup 0 stores dV, warpgroup 1 stores dK (scaled by s)
      const uint32_t t_acc = tmem + lane_off + 256 + D * half;
      const float mul = half == 0 ? 1.0f : p.scale;
      __nv_bfloat16* dst = (half == 0 ? p.dv : p.dk) + (grow * H + u.h) * D;
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += 32) {
        uint32_t o[32];
        tmem_ld32(t_acc + c0, o);
        tmem_ld_wait(o);
        if (row_ok) {
#pragma unroll
          for (int c = 0; c < 32; c += 8) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
              w[e] = pack_bf16(__uint_as_float(o[c + 2 * e]) * mul, __uint_as_float(o[c + 2 * e + 1]) * mul);
            st_global_v4(dst + c0 + c, w[0], w[1], w[2], w[3]);
          }
        }
      }
    } else {
      // warpgroup h stores dQ columns [h D/2, (h+1) D/2), scaled by s (shared
      // queries: fp32 into the per-segment partial rows, summed afterwards)
      const uint32_t t_acc = tmem + lane_off + 256 + (D / 2) * half;
      __nv_bfloat16* dst = p.dq + (grow * H + u.h) * D + (D / 2) * half;
      float* dst32 = p.dq_part + (grow * H + u.h) * D + (D / 2) * half;
#pragma unroll
      for (int c0 = 0; c0 < D / 2; c0 += 16) {
        uint32_t o[16];
        tmem_ld16(t_acc + c0, o);
        tmem_ld_wait16(o);
        if (row_ok) {
          if (p.dq_part) {
#pragma unroll
            for (int c = 0; c < 16; c += 4)
              st_global_v4(dst32 + c0 + c, __float_as_uint(__uint_as_float(o[c]) * p.scale),
                           __float_as_uint(__uint_as_float(o[c + 1]) * p.scale),
                           __float_as_uint(__uint_as_float(o[c + 2]) * p.scale),
                           __float_as_uint(__uint_as_float(o[c + 3]) * p.scale));
          } else {
#pragma unroll
            for (int c = 0; c < 16; c += 8) {
              uint32_t w[4];
#pragma unroll
              for (int e = 0; e < 4; ++e)
                w[e] = pack_bf16(__uint_as_float(o[c + 2 * e]) * p.scale,
                                 __uint_as_float(o[c + 2 * e + 1]) * p.scale);
              st_global_v4(dst + c0 + c, w[0], w[1], w[2], w[3]);
            }
          }
        }
      }
    }
    if constexpr (KV_MAJOR && D <= 64) {
      // fused dQ: this unit's contribution dS K (TMEM lanes are query rows),
      // scaled by s, fp32; warpgroup h writes columns [h D/2, (h+1) D/2)
      if (p.dq_fused != nullptr) {
        const uint32_t t_dq = tmem + lane_off + 256 + 2 * D + (D / 2) * half;
        float* dst = dq_fused_row<D>(p, u, r) + half * (D / 2);
#pragma unroll
        for (int c0 = 0; c0 < D / 2; c0 += 16) {
          uint32_t o[16];
          tmem_ld16(t_dq + c0, o);
          tmem_ld_wait16(o);
          if (r < p.q_rows) {
#pragma unroll
            for (int c = 0; c < 16; c += 4)
              st_global_v4(dst + c0 + c, __float_as_uint(__uint_as_float(o[c]) * p.scale),
                           __float_as_uint(__uint_as_float(o[c + 1]) * p.scale),
                           __float_as_uint(__uint_as_float(o[c + 2]) * p.scale),
                           __float_as_uint(__uint_as_float(o[c + 3]) * p.scale));
          }
        }
      }
    }
    tc_fence_before();
    mbar_arrive_warp(&bars->acc_empty);

    if (want_dbias) {
      // the clamped mass of this unit: one fixed-point red per warp and table
      // end into this CTA's private slice
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        acc_lo += __shfl_xor_sync(0xffffffffu, acc_lo, o);
        acc_hi += __shfl_xor_sync(0xffffffffu, acc_hi, o);
      }
      if ((threadIdx.x & 31) == 0) {
        atomicAdd(part, dbias_fixed(acc_lo));
        atomicAdd(part + 2 * R, dbias_fixed(acc_hi));
      }
    }
  }
  if constexpr (DIRECT && D == 128) {  // this warp's dQ stores are complete before the CTA exits
    if ((threadIdx.x & 31) == 0) bulk_wait_all();
    __syncwarp();
  }
}

// ------------------------------------------------------------------- kernel
template <int D, int ACT, bool KV_MAJOR, bool WIN, bool DIRECT = false>
__global__ void __launch_bounds__(384, 1) gdpa_bwd_kernel(const __grid_constant__ BwdParams p) {
  using C = BwdCfg<D, KV_MAJOR>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  BwdBars* bars = reinterpret_cast<BwdBars*>(smem + C::kBarOff);
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->res_full[i], 1);
      mbar_init(&bars->res_empty[i], 1);
    }
    mbar_init(&bars->s_full, 1);
    mbar_init(&bars->s_free, 8);
    mbar_init(&bars->p_full, 8);
    mbar_init(&bars->dp_full, 1);
    mbar_init(&bars->dp_free, 8);
    mbar_init(&bars->acc_full, 1);
    mbar_init(&bars->acc_empty, 8);
    mbar_init(&bars->drain, 1);
    if constexpr (DIRECT) {
      mbar_init(&bars->dq_full, 1);
      mbar_init(&bars->dq_empty, 8);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars->x_full[s], 8);
      // released by the consuming MMA's commit, plus the dS copy when stored
      mbar_init(&bars->x_empty[s], (KV_MAJOR && p.ds_base != nullptr) ? 2 : 1);
    }
    for (int s = 0; s < 4; ++s) {
      mbar_init(&bars->a_full[s], 1);
      mbar_init(&bars->a_empty[s], 1);
      mbar_init(&bars->b_full[s], 1);
      mbar_init(&bars->b_empty[s], 1);
    }
    bars->abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&bars->tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  int n_units = *p.n_units;
  if (*reinterpret_cast<volatile int*>(p.status) != kOk) n_units = 0;
  Fail fail{&bars->abort, p.status, p.wait_limit_ns};
  if (warp == 0) {
    bwd_producer<D, KV_MAJOR, 0, WIN>(p, smem, bars, n_units, fail);
  } else if (warp == 2) {
    bwd_producer<D, KV_MAJOR, 1, WIN>(p, smem, bars, n_units, fail);
  } else if (warp == 3) {
    if constexpr (KV_MAJOR) {
      if (p.ds_base != nullptr) bwd_ds_store<D, WIN>(p, smem, bars, n_units, fail);
    }
  } else if (warp == 1) {
    if constexpr (KV_MAJOR) bwd_mma_kv<D, WIN, DIRECT>(p, smem, bars, tmem, n_units, fail);
    else bwd_mma_q<D, WIN>(p, smem, bars, tmem, n_units, fail);
  } else if (warp >= 4) {
    bwd_act<D, ACT, KV_MAJOR, WIN, DIRECT>(p, smem, bars, tmem, n_units, fail);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

// ------------------------------------------------ dQ from the stored dS
// dQ pass when the dK/dV pass has stored dS: per unit (segment, head, query
// tile) dQ = s sum_kt dS(qt, kt) K(kt), a plain streaming GEMM.  The stored
// tile is dS^T ([keys][queries]); read as the A operand in MN-major form it
// is dS.  No activation work and no recomputation of S and dP: the pass is
// bound by streaming the dS tiles from memory.
//   warp 0      TMA producer (dS tile + K tile per stage)
//   warp 1      MMA issuer; accumulators double-buffered in TMEM
//   warps 4-7   epilogue (TMEM -> dQ rows)
template <int D>
struct DqCfg : TileCfg<D> {
  using T = TileCfg<D>;
  static constexpr int kStageBytes = kDsTileBytes + T::kTileBytes;
  static constexpr int kStages = D == 128 ? 3 : 4;
  static constexpr int kBarOff = kStages * kStageBytes;
  static constexpr int kSmemBytes = kBarOff + 256 + 1024;
  static_assert(kSmemBytes <= 232448, "shared memory per CTA");
};

struct DqBars {
  uint64_t full[4], empty[4];
  uint64_t acc_full[2], acc_empty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};

template <int D>
__global__ void __launch_bounds__(256, 1) gdpa_dq_ds_kernel(const __grid_constant__ BwdParams p) {
  using C = DqCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  DqBars* bars = reinterpret_cast<DqBars*>(smem + C::kBarOff);
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    for (int s = 0; s < 4; ++s) {
      mbar_init(&bars->full[s], 1);
      mbar_init(&bars->empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars->acc_full[s], 1);
      mbar_init(&bars->acc_empty[s], 4);
    }
    mbar_init(&bars->drain, 1);
    bars->abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&bars->tmem_base, 256);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  int n_units = *p.n_units;
  if (*reinterpret_cast<volatile int*>(p.status) != kOk) n_units = 0;
  Fail fail{&bars->abort, p.status, p.wait_limit_ns};

  if (warp == 0) {  // ---- producer
    const bool leader = elect_one();
    const uint64_t policy = l2_evict_first_policy();  // each dS tile is read once
    uint32_t it = 0;
    bool ok = true;
    for (int r = 0; ok; ++r) {
      const int idx = unit_index(r, blockIdx.x, gridDim.x);
      if (idx >= n_units) break;
      const BwdUnit u = bwd_unit<false, true>(p, idx);
      if (u.rows <= 0) continue;
      for (int i = 0; i < u.count; ++i, ++it) {
        const int kt = u.first + i;
        const int st = it % C::kStages;
        if (!(ok = mbar_wait_warp(&bars->empty[st], ((it / C::kStages) & 1) ^ 1, fail))) break;
        if (leader) {
          uint8_t* dst = smem + st * C::kStageBytes;
          // query rows 64..127 of a tile that ends before them were not
          // stored; their stale half only feeds dQ rows that are not written
          const bool upper = u.rows > kTile / 2;
          mbar_arrive_tx(&bars->full[st], C::kStageBytes - (upper ? 0 : kDsTileBytes / 2));
          const int row = ds_row(p.ds_base, u.seg, u.b, u.h, kt, u.tile, p.window);
          tma_load_2d_hint(dst, &p.tm_ds, &bars->full[st], 0, row, policy);
          if (upper) tma_load_2d_hint(dst + kDsTileBytes / 2, &p.tm_ds, &bars->full[st], kTile / 2, row, policy);
#pragma unroll
          for (int cb = 0; cb < C::kNumBlocks; ++cb)
            tma_load_3d(dst + kDsTileBytes + cb * C::kBlockBytes, &p.tm_k, &bars->full[st], cb * C::kBlockCols,
                        u.h, u.seg.k0 + kt * kTile);
        }
      }
    }
    if (!ok) {
      for (uint32_t i = it > C::kStages ? it - C::kStages : 0; i < it; ++i)
        mbar_wait_drain(&bars->full[i % C::kStages], (i / C::kStages) & 1);
    }
  } else if (warp == 1) {  // ---- MMA issuer
    const bool leader = elect_one();
    constexpr uint32_t idesc = idesc_bf16(kTile, D, 1, 1);  // A (dS) and B (K) MN-major
    uint32_t it = 0, acc_n = 0;
    bool ok = true;
    for (int r = 0; ok; ++r) {
      const int idx = unit_index(r, blockIdx.x, gridDim.x);
      if (idx >= n_units) break;
      const BwdUnit u = bwd_unit<false, true>(p, idx);
      if (u.rows <= 0 || u.count == 0) continue;
      const int buf = acc_n & 1;
      if (!(ok = mbar_wait_warp(&bars->acc_empty[buf], ((acc_n >> 1) & 1) ^ 1, fail))) break;
      const uint32_t d_acc = tmem + buf * D;
      for (int kt = 0; kt < u.count; ++kt, ++it) {
        const int st = it % C::kStages;
        if (!(ok = mbar_wait_warp(&bars->full[st], (it / C::kStages) & 1, fail))) break;
        tc_fence_after();
        const uint32_t a_t = smem_u32(smem + st * C::kStageBytes);
        const uint64_t a0 = mnmajor_desc0<kTile>(a_t), b0 = mnmajor_desc0<D>(a_t + kDsTileBytes);
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk) {
          const uint64_t aoff = static_cast<uint64_t>(kk * 16 * TileCfg<kTile>::kRowBytes) >> 4;
          const uint64_t boff = static_cast<uint64_t>(kk * 16 * C::kRowBytes) >> 4;
          if (leader) mma_ss(d_acc, a0 + aoff, b0 + boff, idesc, (kt > 0 || kk > 0) ? 1u : 0u);
        }
        if (leader) mma_commit(&bars->empty[st]);
      }
      if (!ok) break;
      if (leader) mma_commit(&bars->acc_full[buf]);
      ++acc_n;
    }
    if (leader) mma_commit(&bars->drain);
    mbar_wait_drain(&bars->drain, 0);
  } else if (warp >= 4) {  // ---- epilogue
    const int quad = warp & 3;
    const int r = quad * 32 + (threadIdx.x & 31);
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const int H = p.heads;
    uint32_t acc_n = 0;
    for (int rr = 0;; ++rr) {
      const int idx = unit_index(rr, blockIdx.x, gridDim.x);
      if (idx >= n_units) break;
      const BwdUnit u = bwd_unit<false, true>(p, idx);
      if (u.rows <= 0) continue;
      const bool row_ok = r < u.rows;
      const int64_t grow = static_cast<int64_t>(u.seg.q0) + u.tile * kTile + r;
      __nv_bfloat16* dst = p.dq + (grow * H + u.h) * D;
      float* dst32 = p.dq_part + (grow * H + u.h) * D;  // shared queries: fp32 partial rows
      if (u.count == 0) {  // no keys: zero rows
        if (row_ok) {
          if (p.dq_part) {
#pragma unroll
            for (int c = 0; c < D; c += 4) st_global_v4(dst32 + c, 0u, 0u, 0u, 0u);
          } else {
#pragma unroll
            for (int c = 0; c < D; c += 8) st_global_v4(dst + c, 0u, 0u, 0u, 0u);
          }
        }
        continue;
      }
      const int buf = acc_n & 1;
      if (!mbar_wait(&bars->acc_full[buf], (acc_n >> 1) & 1, fail)) break;
      ++acc_n;
      tc_fence_after();
      const uint32_t t_acc = tmem + lane_off + buf * D;
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += 32) {
        uint32_t o[32];
        tmem_ld32(t_acc + c0, o);
        tmem_ld_wait(o);
        if (row_ok && p.dq_part) {
#pragma unroll
          for (int c = 0; c < 32; c += 4)
            st_global_v4(dst32 + c0 + c, __float_as_uint(__uint_as_float(o[c]) * p.scale),
                         __float_as_uint(__uint_as_float(o[c + 1]) * p.scale),
                         __float_as_uint(__uint_as_float(o[c + 2]) * p.scale),
                         __float_as_uint(__uint_as_float(o[c + 3]) * p.scale));
        } else if (row_ok) {
#pragma unroll
          for (int c = 0; c < 32; c += 8) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
              w[e] = pack_bf16(__uint_as_float(o[c + 2 * e]) * p.scale, __uint_as_float(o[c + 2 * e + 1]) * p.scale);
            st_global_v4(dst + c0 + c, w[0], w[1], w[2], w[3]);
          }
        }
      }
      tc_fence_before();
      mbar_arrive_warp(&bars->acc_empty[buf]);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 256);
}

// delta_i = <dO_i, O_i> per (row, head), fp32 from bf16 (softmax backward).
// D / 16 consecutive lanes share a row: each loads two 16-byte pieces of O
// and of dO (lanes of a group read whole 128-byte lines, a warp 32 / (D / 16)
// rows per load), and the group's partial sums are added by shuffles in a
// fixed order.
template <int D>
__global__ void softmax_delta_kernel(const __nv_bfloat16* __restrict__ out, const __nv_bfloat16* __restrict__ dout,
                                     float* __restrict__ delta, int64_t total_q, int heads, const int* status) {
  constexpr int kLanes = D / 16;  // lanes per (row, head)
  const int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t row = t / kLanes;  // row * heads + h
  const int part = static_cast<int>(t % kLanes);
  if (*status != kOk) return;
  float acc = 0.f;
  if (row < total_q * heads) {
    const uint4* o4 = reinterpret_cast<const uint4*>(out + row * D);
    const uint4* d4 = reinterpret_cast<const uint4*>(dout + row * D);
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const uint4 a = __ldg(o4 + part + k * kLanes), b = __ldg(d4 + part + k * kLanes);
      const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, bw[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        acc = __fmaf_rn(__uint_as_float(aw[e] << 16), __uint_as_float(bw[e] << 16), acc);
        acc = __fmaf_rn(__uint_as_float(aw[e] & 0xFFFF0000u), __uint_as_float(bw[e] & 0xFFFF0000u), acc);
      }
    }
  }
#pragma unroll
  for (int o = kLanes / 2; o > 0; o >>= 1) acc += __shfl_down_sync(0xffffffffu, acc, o, kLanes);
  if (part == 0 && row < total_q * heads) {
    const int64_t tq = row / heads, h = row % heads;
    delta[h * total_q + tq] = acc;
  }
}

#if JGDPA_HEAD_DIM == 128
// dbias[h][e] = sum over CTAs of the per-CTA fixed-point partial sums
// (exact integer additions), converted to fp32 once.
__global__ void dbias_reduce_kernel(const unsigned long long* __restrict__ part, float* __restrict__ dbias,
                                    int n_parts, int n) {
  const int e = blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= n) return;
  unsigned long long acc = 0;
  for (int c = 0; c < n_parts; ++c) acc += part[static_cast<int64_t>(c) * n + e];
  dbias[e] = static_cast<float>(static_cast<double>(static_cast<long long>(acc)) *
                                (1.0 / static_cast<double>(1ll << kDbiasFracBits)));
}
#endif

// ------------------------------------------------------------------- launch
// Each object file holds the kernels of one head dimension (JGDPA_HEAD_DIM),
// so that the build compiles the head dimensions in parallel; the
// head-dimension-free dbias reduction lives in the d = 128 object.
#ifndef JGDPA_HEAD_DIM
#error "compile bwd.cu with -DJGDPA_HEAD_DIM=32, 64 or 128"
#endif

template <int D, int ACT, bool KV_MAJOR, bool DIRECT = false>
static cudaError_t launch_bwd_t(const BwdParams& p, int grid, cudaStream_t stream) {
  using C = BwdCfg<D, KV_MAJOR>;
  decltype(&gdpa_bwd_kernel<D, ACT, KV_MAJOR, false>) kern;
  if constexpr (DIRECT) kern = gdpa_bwd_kernel<D, ACT, true, false, true>;  // (direct-dQ segments: no window)
  else kern = p.window > 0 ? gdpa_bwd_kernel<D, ACT, KV_MAJOR, true> : gdpa_bwd_kernel<D, ACT, KV_MAJOR, false>;
  static DeviceFlags attr_set[2] = {};
  cudaError_t e = smem_attr_once(kern, C::kSmemBytes, attr_set[!DIRECT && p.window > 0]);
  if (e != cudaSuccess) return e;
  kern<<<grid, 384, C::kSmemBytes, stream>>>(p);
  return cudaGetLastError();
}

// direct: the key-major pass over the direct-dQ segments' units (DIRECT).
template <int D>
cudaError_t launch_bwd_pass_d(const BwdParams& p, int act, bool kv_major, int grid, cudaStream_t stream,
                              bool direct) {
  if (direct) {
    if (act == 0) return launch_bwd_t<D, 0, true, true>(p, grid, stream);
    if (act == 1) return launch_bwd_t<D, 1, true, true>(p, grid, stream);
    return launch_bwd_t<D, 2, true, true>(p, grid, stream);
  }
  if (kv_major) {
    if (act == 0) return launch_bwd_t<D, 0, true>(p, grid, stream);
    if (act == 1) return launch_bwd_t<D, 1, true>(p, grid, stream);
    return launch_bwd_t<D, 2, true>(p, grid, stream);
  }
  if (act == 0) return launch_bwd_t<D, 0, false>(p, grid, stream);
  if (act == 1) return launch_bwd_t<D, 1, false>(p, grid, stream);
  return launch_bwd_t<D, 2, false>(p, grid, stream);
}
template cudaError_t launch_bwd_pass_d<JGDPA_HEAD_DIM>(const BwdParams&, int, bool, int, cudaStream_t, bool);

template <int D>
cudaError_t launch_dq_ds_d(const BwdParams& p, int grid, cudaStream_t stream) {
  using C = DqCfg<D>;
  auto kern = gdpa_dq_ds_kernel<D>;
  static DeviceFlags attr_set = {};
  cudaError_t e = smem_attr_once(kern, C::kSmemBytes, attr_set);
  if (e != cudaSuccess) return e;
  kern<<<grid, 256, C::kSmemBytes, stream>>>(p);
  return cudaGetLastError();
}
template cudaError_t launch_dq_ds_d<JGDPA_HEAD_DIM>(const BwdParams&, int, cudaStream_t);

template <int D>
cudaError_t launch_softmax_delta_d(const void* out, const void* dout, float* delta, int64_t total_q, int heads,
                                   const int* status, cudaStream_t stream) {
  const int64_t rows = total_q * heads;
  if (rows == 0) return cudaSuccess;
  const int threads = 256;
  const int64_t lanes = rows * (D / 16);
  const unsigned blocks = static_cast<unsigned>((lanes + threads - 1) / threads);
  softmax_delta_kernel<D><<<blocks, threads, 0, stream>>>(static_cast<const __nv_bfloat16*>(out),
                                                          static_cast<const __nv_bfloat16*>(dout), delta, total_q,
                                                          heads, status);
  return cudaGetLastError();
}
template cudaError_t launch_softmax_delta_d<JGDPA_HEAD_DIM>(const void*, const void*, float*, int64_t, int,
                                                            const int*, cudaStream_t);

#if JGDPA_HEAD_DIM == 128
// Shared queries: dq[s][h][c] = sum over segments b (in order) of the fp32
// partial dQ rows part[b S + s][h][c], rounded to bf16 once.
__global__ void dq_shared_reduce_kernel(const float* __restrict__ part, __nv_bfloat16* __restrict__ dq,
                                        int batch, int64_t n, const int* status) {
  const int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;  // (s, h, c) of [S][H][D]
  if (e >= n || *status != kOk) return;
  float acc = 0.f;
  for (int b = 0; b < batch; ++b) acc += part[static_cast<int64_t>(b) * n + e];
  dq[e] = __float2bfloat16_rn(acc);
}

cudaError_t launch_dq_shared_reduce(const float* part, void* dq, int batch, int64_t n, const int* status,
                                    cudaStream_t stream) {
  if (n == 0) return cudaSuccess;
  dq_shared_reduce_kernel<<<static_cast<unsigned>((n + 255) / 256), 256, 0, stream>>>(
      part, static_cast<__nv_bfloat16*>(dq), batch, n, status);
  return cudaGetLastError();
}

// Fused dQ of shared queries: dq[s][h][c] = sum over key items i (in item
// order) of the blocks part[i H + h][s][c].  Stage 1: kFusedChunks threads
// per element each sum a contiguous, fixed range of items into tmp; stage 2
// sums those in chunk order and rounds once.  The item count is read from the
// scheduler's prefix (item_base[batch]); the split depends only on it, so
// the result is the same bit for bit on every run.
constexpr int kFusedChunks = 64;
__global__ void dq_fused_stage1_kernel(const float* __restrict__ part, float* __restrict__ tmp,
                                       const int32_t* __restrict__ item_base, int batch, int heads, int rows,
                                       int d, const int* status) {
  const int64_t per = static_cast<int64_t>(rows) * heads * d;  // elements of dq
  const int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (t >= per * kFusedChunks || *status != kOk) return;
  const int chunk = static_cast<int>(t / per);
  const int64_t e = t % per;  // (s, h, c) of [S][H][D]
  const int s_row = static_cast<int>(e / (static_cast<int64_t>(heads) * d));
  const int h = static_cast<int>((e / d) % heads), c = static_cast<int>(e % d);
  const int n_items = item_base[batch];
  const int len = (n_items + kFusedChunks - 1) / kFusedChunks;
  const int i0 = chunk * len, i1 = min(n_items, i0 + len);
  float acc = 0.f;
  for (int i = i0; i < i1; ++i)
    acc += part[((static_cast<int64_t>(i) * heads + h) * rows + s_row) * d + c];
  tmp[t] = acc;
}
__global__ void dq_fused_stage2_kernel(const float* __restrict__ tmp, __nv_bfloat16* __restrict__ dq, int64_t per,
                                       const int* status) {
  const int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (e >= per || *status != kOk) return;
  float acc = 0.f;
  for (int k = 0; k < kFusedChunks; ++k) acc += tmp[static_cast<int64_t>(k) * per + e];
  dq[e] = __float2bfloat16_rn(acc);
}

cudaError_t launch_dq_fused_reduce(const float* part, float* tmp, void* dq, const int32_t* item_base, int batch,
                                   int heads, int rows, int d, const int* status, cudaStream_t stream) {
  const int64_t per = static_cast<int64_t>(rows) * heads * d;
  if (per == 0) return cudaSuccess;
  dq_fused_stage1_kernel<<<static_cast<unsigned>((per * kFusedChunks + 255) / 256), 256, 0, stream>>>(
      part, tmp, item_base, batch, heads, rows, d, status);
  dq_fused_stage2_kernel<<<static_cast<unsigned>((per + 255) / 256), 256, 0, stream>>>(
      tmp, static_cast<__nv_bfloat16*>(dq), per, status);
  return cudaGetLastError();
}
size_t dq_fused_tmp_floats(int heads, int rows, int d) {
  return static_cast<size_t>(kFusedChunks) * rows * heads * d;
}

cudaError_t launch_dbias_reduce(const unsigned long long* part, float* dbias, int n_parts, int n,
                                cudaStream_t stream) {
  if (n == 0) return cudaSuccess;
  dbias_reduce_kernel<<<(n + 255) / 256, 256, 0, stream>>>(part, dbias, n_parts, n);
  return cudaGetLastError();
}
#endif

}  // namespace jg
