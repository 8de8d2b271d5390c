// Forward jagged GDPA kernel for sm_103a.
//
// A persistent CTA (one per SM) walks the scheduler's unit list.  A unit is a
// (segment b, head h, pair of 128-row query tiles); the two query tiles share
// every key/value tile of the segment.  Warp roles:
//   warp 0      TMA producer: Q tiles into two slots, K/V tiles into a ring
//   warp 1      MMA issuer (one thread): S = Q K^T and O += P V with tcgen05,
//               accumulators in Tensor Memory; also owns the TMEM allocation
//   warps 4-7   activation warpgroup of query slot 0
//   warps 8-11  activation warpgroup of query slot 1
// The two slots ping-pong: while one warpgroup turns S into P the tensor core
// works on the other slot, so activation and MMA overlap.
//
// TMEM columns: S0/P0 [0,128), S1/P1 [128,256), O0 [256,256+D),
// O1 [256+D, 256+2D).  P (bf16) is written over the first 64 columns of its
// S and consumed from TMEM by the second MMA.
//
// GELU/SiLU mode has no normalisation and no online rescaling: O accumulates
// in TMEM over every key/value tile and is stored once (the "softmax
// correction stage elimination" of the GDPA redesign, aiuniverse.news,
// section "Custom Kernels and 5D Parallelism ...").  Softmax mode (Jagged
// Flash Attention) keeps a running row maximum in base 2 and rescales O in
// TMEM only when the maximum grows by more than 2^8.
//
// Masking follows the jagged "subtraction scheme" ("Eliminating Compute Waste
// in Asymmetric Workloads", aiuniverse.news): per tile and row the number of
// valid columns n = min(Lkv - j0, causal ? i - j0 + 1 : 128) is computed once,
// and only tiles where n < 128 compare column indices against it.
#include "act.cuh"
#include "common.cuh"
#include "ptx.cuh"

namespace jg {

// Routes of the four 32-column chunks of every S tile: the last
// JGDPA_FWD_ALU_CHUNKS take the ALU polynomial route, the
// JGDPA_FWD_EX2_CHUNKS before them the ex2 route, the rest the hardware tanh.
// Measured on GB300 (long-tail workload, d = 128, GELU): every chunk moved
// off the tanh route made the forward slower (0/1/3/4 ex2 chunks:
// 2.83/3.06/3.49/3.85 ms on an earlier build; 0/1/2 ALU chunks: 2.63/3.01/
// 3.63 ms), so both default to 0 and the other routes stay available as
// compile-time options.
#ifndef JGDPA_FWD_ALU_CHUNKS
#define JGDPA_FWD_ALU_CHUNKS 0
#endif
#ifndef JGDPA_FWD_EX2_CHUNKS
#define JGDPA_FWD_EX2_CHUNKS 0
#endif
constexpr int kFwdAluChunks = JGDPA_FWD_ALU_CHUNKS;
constexpr int kFwdEx2Chunks = JGDPA_FWD_EX2_CHUNKS;
static_assert(kFwdAluChunks + kFwdEx2Chunks <= 4, "four 32-column chunks per tile");

template <int D>
struct FwdCfg {
  static constexpr int kBlockCols = D < 64 ? D : 64;      // bf16 columns per swizzle row
  static constexpr int kRowBytes = kBlockCols * 2;        // 64 or 128 bytes
  static constexpr int kBlockBytes = kTile * kRowBytes;   // one column block of a tile
  static constexpr int kNumBlocks = D / kBlockCols;
  static constexpr int kTileBytes = kTile * D * 2;
  static constexpr int kStages = D == 128 ? 2 : 4;
  static constexpr uint32_t kSwizzle = kRowBytes == 128 ? 2u : 4u;  // 128-byte / 64-byte
  static constexpr int kSBO = 8 * kRowBytes;              // stride between 8-row groups
  static constexpr int kQOff = 0;
  static constexpr int kKOff = kQOff + 2 * kTileBytes;
  static constexpr int kVOff = kKOff + kStages * kTileBytes;
  static constexpr int kEpiOff = kVOff + kStages * kTileBytes;  // epilogue staging, if any
  static constexpr int kTmemCols = 512;
};

// The rest of the layout depends on the activation: GELU / SiLU at d >= 64
// stage the O epilogue (4 KB per activation warp).  Softmax does not: its
// kernel spills more, spills go through L1, and L1 is what shared memory
// leaves over (the staged softmax forward measured 8% slower).
template <int D, int ACT>
struct FwdSmem {
  static constexpr bool kStage = D >= 64 && ACT != 2;
  static constexpr int kBarOff = FwdCfg<D>::kEpiOff + (kStage ? 8 * 4096 : 0);
  static constexpr int kSmemBytes = kBarOff + 512 + 1024;  // + barriers + alignment slack
  static_assert(kSmemBytes <= 232448, "shared memory per CTA");
};

struct FwdBars {
  uint64_t q_full[2], q_empty[2];
  uint64_t s_full[2], p_full[2], o_full[2], o_empty[2];
  uint64_t drain;
  uint64_t k_full[4], k_empty[4], v_full[4], v_empty[4];
  uint32_t tmem_base;
  int abort;
};

// Per-unit geometry shared by every role.
// The unit streams key/value tiles k0 .. k0 + nkv - 1 once; query slot s
// uses stream positions [beg_s, beg_s + nkv_s) of it (the two query tiles'
// spans overlap or touch, so their union has no gap).
struct FwdUnit {
  int b, h, pair;
  Seg seg;
  int k0;         // first key/value tile of the stream
  int nkv;        // tiles streamed
  int beg_s[2];   // each query slot's first stream position
  int nkv_s[2];   // key/value tiles for each query slot (0 = slot idle)
  int rows_s[2];  // valid query rows in each slot's tile (<= 0: no tile)
};

// WIN: the kernel is compiled for a sliding window (p.window > 0); the plain
// kernels fold the window away.
template <bool WIN>
__device__ __forceinline__ FwdUnit fwd_unit(const FwdParams& p, int idx) {
  const int window = WIN ? p.window : 0;
  FwdUnit u;
  const Unit w = p.units[idx];
  u.b = w.x;
  u.h = w.y;
  u.pair = w.z;
  u.seg = load_seg(p.q_off, p.kv_off, u.b);
  int lo = 0x7fffffff, hi = 0;
  int first[2];
#pragma unroll
  for (int s = 0; s < 2; ++s) {
    const int t = 2 * u.pair + s;
    u.rows_s[s] = u.seg.lq - t * kTile;
    const TileSpan sp = u.rows_s[s] > 0 ? kv_span_for_q_tile(t, u.seg.lkv, p.causal, window) : TileSpan{0, 0};
    u.nkv_s[s] = sp.count;
    first[s] = sp.first;
    if (sp.count > 0) {
      lo = min(lo, sp.first);
      hi = max(hi, sp.first + sp.count);
    }
  }
  u.k0 = hi > 0 ? lo : 0;
  u.nkv = hi > 0 ? hi - lo : 0;
#pragma unroll
  for (int s = 0; s < 2; ++s) u.beg_s[s] = first[s] - u.k0;
  return u;
}

// --------------------------------------------------------------- producer
template <int D, bool WIN>
__device__ void fwd_producer(const FwdParams& p, uint8_t* smem, FwdBars* bars, int n_units, Fail fail) {
  using C = FwdCfg<D>;
  uint32_t q_it[2] = {0, 0};
  uint32_t kv_it = 0;  // K/V stream positions whose V load was issued
  uint32_t k_it = 0;   // K loads issued (one ahead of kv_it if a V wait failed)
  const bool leader = elect_one();
  bool ok = true;
  for (int r = 0;; ++r) {
    const int idx = unit_index(r, blockIdx.x, gridDim.x);
    if (idx >= n_units) break;
    const FwdUnit u = fwd_unit<WIN>(p, idx);
    if (u.nkv == 0) continue;
    for (int s = 0; s < 2 && ok; ++s) {
      if (u.nkv_s[s] == 0) continue;
      ok = mbar_wait_warp(&bars->q_empty[s], (q_it[s] & 1) ^ 1, fail);
      if (!ok) break;
      if (leader) {
        mbar_arrive_tx(&bars->q_full[s], C::kTileBytes);
        uint8_t* dst = smem + C::kQOff + s * C::kTileBytes;
        // shared queries: the Q map holds the shared rows once
        const int row = (p.q_shared ? 0 : u.seg.q0) + (2 * u.pair + s) * kTile;
#pragma unroll
        for (int cb = 0; cb < C::kNumBlocks; ++cb)
          tma_load_3d(dst + cb * C::kBlockBytes, &p.tm_q, &bars->q_full[s], cb * C::kBlockCols, u.h, row);
      }
      ++q_it[s];
    }
    // K and V of a stage are released separately (K after the last S that
    // reads it, V after the last P V), so K loads run well ahead of use.
    for (int kt = 0; kt < u.nkv && ok; ++kt) {
      const int st = kv_it % C::kStages;
      const uint32_t empty_phase = ((kv_it / C::kStages) & 1) ^ 1;
      if (!(ok = mbar_wait_warp(&bars->k_empty[st], empty_phase, fail))) break;
      const int row = u.seg.k0 + (u.k0 + kt) * kTile;
      if (leader) {
        mbar_arrive_tx(&bars->k_full[st], C::kTileBytes);
        uint8_t* kd = smem + C::kKOff + st * C::kTileBytes;
#pragma unroll
        for (int cb = 0; cb < C::kNumBlocks; ++cb)
          tma_load_3d(kd + cb * C::kBlockBytes, &p.tm_k, &bars->k_full[st], cb * C::kBlockCols, u.h, row);
      }
      ++k_it;
      if (!(ok = mbar_wait_warp(&bars->v_empty[st], empty_phase, fail))) break;
      if (leader) {
        mbar_arrive_tx(&bars->v_full[st], C::kTileBytes);
        uint8_t* vd = smem + C::kVOff + st * C::kTileBytes;
#pragma unroll
        for (int cb = 0; cb < C::kNumBlocks; ++cb)
          tma_load_3d(vd + cb * C::kBlockBytes, &p.tm_v, &bars->v_full[st], cb * C::kBlockCols, u.h, row);
      }
      ++kv_it;
    }
    if (!ok) break;
  }
  if (!ok) {
    // Let copies already issued land before the CTA exits.
    for (int s = 0; s < 2; ++s)
      if (q_it[s]) mbar_wait_drain(&bars->q_full[s], (q_it[s] - 1) & 1);
    for (uint32_t i = k_it > C::kStages ? k_it - C::kStages : 0; i < k_it; ++i)
      mbar_wait_drain(&bars->k_full[i % C::kStages], (i / C::kStages) & 1);
    for (uint32_t i = kv_it > C::kStages ? kv_it - C::kStages : 0; i < kv_it; ++i)
      mbar_wait_drain(&bars->v_full[i % C::kStages], (i / C::kStages) & 1);
  }
}

// ------------------------------------------------------------- MMA issuer
// The MMA helpers are called by the whole MMA warp (descriptors are
// warp-uniform); `leader` issues.
template <int D>
__device__ __forceinline__ void issue_qk(uint32_t tmem_s, uint32_t q_addr, uint32_t k_addr, bool leader) {
  using C = FwdCfg<D>;
  constexpr uint32_t idesc = idesc_bf16(kTile, kTile, 0, 0);
  const uint64_t a0 = sdesc(q_addr, 16, C::kSBO, C::kSwizzle), b0 = sdesc(k_addr, 16, C::kSBO, C::kSwizzle);
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint64_t off = static_cast<uint64_t>((kk * 16 / C::kBlockCols) * C::kBlockBytes + (kk * 16 % C::kBlockCols) * 2) >> 4;
    if (leader) mma_ss(tmem_s, a0 + off, b0 + off, idesc, kk > 0 ? 1u : 0u);
  }
}

template <int D>
__device__ __forceinline__ void issue_pv(uint32_t tmem_o, uint32_t tmem_p, uint32_t v_addr, bool accumulate,
                                         bool leader) {
  using C = FwdCfg<D>;
  constexpr uint32_t idesc = idesc_bf16(kTile, D, 0, 1);  // B (= V) is MN-major
  const uint64_t b0 = sdesc(v_addr, C::kBlockBytes, C::kSBO, C::kSwizzle);
#pragma unroll
  for (int kk = 0; kk < kTile / 16; ++kk) {
    const uint64_t off = static_cast<uint64_t>(kk * 16 * C::kRowBytes) >> 4;
    if (leader) mma_ts(tmem_o, tmem_p + kk * 8, b0 + off, idesc, (accumulate || kk > 0) ? 1u : 0u);
  }
}

template <int D, bool WIN>
__device__ void fwd_mma(const FwdParams& p, uint8_t* smem, FwdBars* bars, uint32_t tmem, int n_units, Fail fail) {
  using C = FwdCfg<D>;
  const uint32_t q_addr[2] = {smem_u32(smem + C::kQOff), smem_u32(smem + C::kQOff + C::kTileBytes)};
  const uint32_t k_base = smem_u32(smem + C::kKOff);
  const uint32_t v_base = smem_u32(smem + C::kVOff);
  const uint32_t t_s[2] = {tmem, tmem + 128};
  const uint32_t t_o[2] = {tmem + 256, tmem + 256 + D};
  uint32_t q_it[2] = {0, 0}, p_it[2] = {0, 0}, o_it[2] = {0, 0};
  uint32_t kv_it = 0;
  const bool leader = elect_one();
  bool ok = true;

  for (int r = 0; ok; ++r) {
    const int idx = unit_index(r, blockIdx.x, gridDim.x);
    if (idx >= n_units) break;
    const FwdUnit u = fwd_unit<WIN>(p, idx);
    if (u.nkv == 0) continue;
    for (int s = 0; s < 2 && ok; ++s) {
      if (u.nkv_s[s] == 0) continue;
      ok = mbar_wait_warp(&bars->q_full[s], q_it[s] & 1, fail);
      ++q_it[s];
    }
    if (!ok) break;
    // slot s takes stream positions [b_s, e_s)
    const int b0 = u.beg_s[0], e0 = b0 + u.nkv_s[0];
    const int b1 = u.beg_s[1], e1 = b1 + u.nkv_s[1];
    // S of stream position 0 for the slots that start there
    {
      const int st = kv_it % C::kStages;
      if (!(ok = mbar_wait_warp(&bars->k_full[st], (kv_it / C::kStages) & 1, fail))) break;
      tc_fence_after();
      for (int s = 0; s < 2; ++s) {
        if (u.nkv_s[s] == 0 || u.beg_s[s] != 0) continue;
        issue_qk<D>(t_s[s], q_addr[s], k_base + st * C::kTileBytes, leader);
        if (leader) mma_commit(&bars->s_full[s]);
        if (u.nkv_s[s] == 1) if (leader) mma_commit(&bars->q_empty[s]);
      }
      if (leader) mma_commit(&bars->k_empty[st]);  // every S of stream position 0 issued
    }
    for (int kt = 0; kt < u.nkv && ok; ++kt) {
      const uint32_t it = kv_it + kt;
      const int st = it % C::kStages;
      const uint32_t v_addr = v_base + st * C::kTileBytes;
      if (!(ok = mbar_wait_warp(&bars->v_full[st], (it / C::kStages) & 1, fail))) break;
      const bool more = kt + 1 < u.nkv;
      const int st1 = (it + 1) % C::kStages;
      // Order per tile: PV0(kt), S0(kt+1), PV1(kt), S1(kt+1).  Each slot's
      // activation then has the other slot's PV and S (two MMA groups) to
      // hide behind.  S_s(kt+1) overwrites the columns that PV_s(kt) reads;
      // it is issued after it, and MMAs execute in issue order.
      // slot 0: O0 += P0 V, then S0 of the next tile
      if (kt >= b0 && kt < e0) {
        if (kt == b0) {
          if (!(ok = mbar_wait_warp(&bars->o_empty[0], (o_it[0] & 1) ^ 1, fail))) break;
          ++o_it[0];
        }
        if (!(ok = mbar_wait_warp(&bars->p_full[0], p_it[0] & 1, fail))) break;
        ++p_it[0];
        tc_fence_after();
        issue_pv<D>(t_o[0], t_s[0], v_addr, kt > b0, leader);
        if (kt == e0 - 1) if (leader) mma_commit(&bars->o_full[0]);
      }
      if (more) {
        if (!(ok = mbar_wait_warp(&bars->k_full[st1], ((it + 1) / C::kStages) & 1, fail))) break;
        tc_fence_after();
        if (kt + 1 >= b0 && kt + 1 < e0) {
          issue_qk<D>(t_s[0], q_addr[0], k_base + st1 * C::kTileBytes, leader);
          if (leader) mma_commit(&bars->s_full[0]);
          if (kt + 1 == e0 - 1) if (leader) mma_commit(&bars->q_empty[0]);
        }
      }
      // slot 1: O1 += P1 V, release V, then S1 of the next tile, release K
      if (kt >= b1 && kt < e1) {
        if (kt == b1) {
          if (!(ok = mbar_wait_warp(&bars->o_empty[1], (o_it[1] & 1) ^ 1, fail))) break;
          ++o_it[1];
        }
        if (!(ok = mbar_wait_warp(&bars->p_full[1], p_it[1] & 1, fail))) break;
        ++p_it[1];
        tc_fence_after();
        issue_pv<D>(t_o[1], t_s[1], v_addr, kt > b1, leader);
        if (kt == e1 - 1) if (leader) mma_commit(&bars->o_full[1]);
      }
      if (leader) mma_commit(&bars->v_empty[st]);  // every P V of V(kt) issued
      if (more && kt + 1 >= b1 && kt + 1 < e1) {
        issue_qk<D>(t_s[1], q_addr[1], k_base + st1 * C::kTileBytes, leader);
        if (leader) mma_commit(&bars->s_full[1]);
        if (kt + 1 == e1 - 1) if (leader) mma_commit(&bars->q_empty[1]);
      }
      if (more) if (leader) mma_commit(&bars->k_empty[st1]);  // every S of K(kt+1) issued
    }
    kv_it += u.nkv;
  }
  // Make sure every MMA issued so far has finished before TMEM is released.
  if (leader) mma_commit(&bars->drain);
  mbar_wait_drain(&bars->drain, 0);
}

// ------------------------------------------------------ activation warps
// Per tile, the thread of row r (query i = i0 + r) and column c (key
// j = j0 + c) has rel = i - j = (i0 - j0) + r - c and bias index
// clamp(rel, -R, R) + R = clamp(base - c, 0, 2R) with base = i0 - j0 + r + R.
// A tile whose rel range lies wholly at or beyond +-R uses one constant, so
// only the few tiles near the diagonal look the table up per element.
struct TileBias {
  bool band;          // per-element lookups needed
  float value;        // the constant otherwise (0 without a table)
  int base;           // base for band tiles
  int top;            // 2R
  const float* row;   // this head's table
};

// bc_lo / bc_hi: the head's two end entries, loaded once per unit.
__device__ __forceinline__ TileBias tile_bias(const FwdParams& p, int h, int i0, int r, int j0, float bc_lo,
                                              float bc_hi) {
  TileBias t{false, 0.f, 0, p.bias_len - 1, nullptr};
  if (p.bias_len == 0) return t;
  const int R = (p.bias_len - 1) / 2;
  const int delta = i0 - j0;
  t.row = p.bias + static_cast<int64_t>(h) * p.bias_len;
  if (delta - (kTile - 1) >= R) {
    t.value = bc_hi;
  } else if (delta + (kTile - 1) <= -R) {
    t.value = bc_lo;
  } else {
    t.band = true;
    t.base = delta + r + R;
  }
  return t;
}

__device__ __forceinline__ float2 band_bias2(const TileBias& tb, int c, float mul) {
  return make_float2(mul * ld_nc_f32(tb.row + min(max(tb.base - c, 0), tb.top)),
                     mul * ld_nc_f32(tb.row + min(max(tb.base - c - 1, 0), tb.top)));
}

// S (fp32, TMEM) -> P = act(s S + bias) (bf16, over the same TMEM columns)
// for one 128 x 128 tile, GELU / SiLU, two columns per packed instruction.
// The last NALU of the four 32-column chunks take the ALU route.  MASKED:
// columns outside [lo, nvalid) (nvalid: the subtraction-scheme count; lo > 0
// only under a sliding window) get P = act(0) = 0.
// The four 32-column chunks are software-pipelined: the TMEM load of chunk
// q + 1 is in flight while chunk q is computed and its P stored (P of chunk q
// lands in columns [16q, 16q + 16), all read already).
// nchunks (>= 1, the same for every thread): 32-column chunks that hold a
// key row of the segment; the rest are not computed, and their P is zero (the
// PV product reads every column).
template <int ACT, int NALU, bool BAND, bool MASKED>
__device__ __forceinline__ void tile_act(uint32_t t_s, float hs, const TileBias& tb, int lo, int nvalid,
                                         int nchunks) {
  const float hb = 0.5f * tb.value;
  uint32_t buf0[32], buf1[32];
  tmem_ld32(t_s, buf0);
  tmem_ld_wait(buf0);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint32_t(&cur)[32] = (q & 1) ? buf1 : buf0;
    uint32_t(&nxt)[32] = (q & 1) ? buf0 : buf1;
    if (q < 3) tmem_ld32(t_s + 32 * (q + 1), nxt);
    uint32_t pk[16];
    if (MASKED && q >= nchunks) {
#pragma unroll
      for (int c2 = 0; c2 < 16; ++c2) pk[c2] = 0u;
    } else {
  #pragma unroll
      for (int c2 = 0; c2 < 16; ++c2) {
        const int c = 32 * q + 2 * c2;
        const float2 sv = make_float2(__uint_as_float(cur[2 * c2]), __uint_as_float(cur[2 * c2 + 1]));
        const float2 bias = BAND ? band_bias2(tb, c, 0.5f) : f2(hb);
        float2 hx = __ffma2_rn(sv, f2(hs), bias);  // x / 2
        if (MASKED) {
          if (c < lo || c >= nvalid) hx.x = 0.f;
          if (c + 1 < lo || c + 1 >= nvalid) hx.y = 0.f;
        }
        float2 y;
        if (q >= 4 - NALU) y = act2_route<ACT, 1>(hx);
        else if (q >= 4 - NALU - kFwdEx2Chunks) y = act2_route<ACT, 2>(hx);
        else y = act2_route<ACT, 0>(hx);
        pk[c2] = pack_bf16(y.x, y.y);
      }
    }
    tmem_st16(t_s + 16 * q, pk);
    if (q < 3) tmem_ld_wait(nxt);
  }
}

// Softmax tile (base 2): x2 = (s S + bias) log2 e, row maximum, lazy rescale
// of O (only when the maximum grows by more than 8, i.e. a factor 256),
// P = 2^(x2 - m) over the S columns, running row sum.
template <int D, bool BAND, bool MASKED>
__device__ __forceinline__ void tile_softmax(uint32_t t_s, uint32_t t_o, float scale2, const TileBias& tb,
                                             int lo, int nvalid, bool first, float& m_run, float& l_run) {
  uint32_t a[32], b[32], c3[32], d4[32];
  tmem_ld32(t_s, a);
  tmem_ld32(t_s + 32, b);
  tmem_ld_wait2(a, b);
  tmem_ld32(t_s + 64, c3);
  tmem_ld32(t_s + 96, d4);
  tmem_ld_wait2(c3, d4);
  const float b2 = kLog2e * tb.value;
  float mx = -INFINITY;
#pragma unroll
  for (int c = 0; c < 128; c += 2) {
    uint32_t& r0 = c < 32 ? a[c] : c < 64 ? b[c - 32] : c < 96 ? c3[c - 64] : d4[c - 96];
    uint32_t& r1 = c < 32 ? a[c + 1] : c < 64 ? b[c - 31] : c < 96 ? c3[c - 63] : d4[c - 95];
    const float2 bias = BAND ? band_bias2(tb, c, kLog2e) : f2(b2);
    float2 x = __ffma2_rn(make_float2(__uint_as_float(r0), __uint_as_float(r1)), f2(scale2), bias);
    if (MASKED) {
      if (c < lo || c >= nvalid) x.x = -INFINITY;
      if (c + 1 < lo || c + 1 >= nvalid) x.y = -INFINITY;
    }
    r0 = __float_as_uint(x.x);
    r1 = __float_as_uint(x.y);
    mx = fmaxf(mx, fmaxf(x.x, x.y));
  }
  const bool grow_max = mx > m_run + 8.0f;
  const float m_new = grow_max ? mx : m_run;
  const float factor = grow_max ? ex2_sfu(m_run - m_new) : 1.0f;  // ex2(-inf) = 0 on the first tile
  l_run *= factor;
  m_run = m_new;
  float2 lsum = f2(0.f);
  // a row with no key so far (a sliding window can leave whole tiles empty
  // for it) keeps m = -inf; its x are all -inf and P must come out 0
  const float2 neg_m = f2(m_run == -INFINITY ? 0.f : -m_run);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint32_t(&src)[32] = q == 0 ? a : q == 1 ? b : q == 2 ? c3 : d4;
    uint32_t pk[16];
#pragma unroll
    for (int c2 = 0; c2 < 16; ++c2) {
      const float2 z =
          __fadd2_rn(make_float2(__uint_as_float(src[2 * c2]), __uint_as_float(src[2 * c2 + 1])), neg_m);
      const float2 pv = make_float2(ex2_sfu(z.x), ex2_sfu(z.y));
      lsum = __fadd2_rn(lsum, pv);
      pk[c2] = pack_bf16(pv.x, pv.y);
    }
    tmem_st16(t_s + 16 * q, pk);  // P columns [16q, 16q+16) lie in S columns already read
  }
  l_run += lsum.x + lsum.y;
  // O holds every earlier tile's P V (complete: it was issued before this
  // tile's S), so it can be rescaled in place before P is released.
  if (!first && __any_sync(0xffffffffu, grow_max)) {
#pragma unroll
    for (int c0 = 0; c0 < D; c0 += 32) {
      uint32_t o[32];
      tmem_ld32(t_o + c0, o);
      tmem_ld_wait(o);
#pragma unroll
      for (int i = 0; i < 32; i += 2) {
        const float2 v = __fmul2_rn(make_float2(__uint_as_float(o[i]), __uint_as_float(o[i + 1])), f2(factor));
        o[i] = __float_as_uint(v.x);
        o[i + 1] = __float_as_uint(v.y);
      }
      tmem_st32(t_o + c0, o);
    }
  }
}

template <int D, int ACT, int NALU, bool WIN>
__device__ void fwd_act(const FwdParams& p, uint8_t* smem, FwdBars* bars, uint32_t tmem, int slot, int n_units,
                        Fail fail) {
  using C = FwdCfg<D>;
  constexpr bool kSoftmax = ACT == 2;
  const int warp = threadIdx.x >> 5;
  const int quad = warp & 3;
  const int r = quad * 32 + (threadIdx.x & 31);  // row of the tile owned by this thread
  const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
  const uint32_t t_s = tmem + lane_off + 128 * slot;
  const uint32_t t_o = tmem + lane_off + 256 + D * slot;
  uint32_t s_it = 0, o_it = 0;
  const int H = p.heads;

  for (int rr = 0;; ++rr) {
    const int idx = unit_index(rr, blockIdx.x, gridDim.x);
    if (idx >= n_units) break;
    const FwdUnit u = fwd_unit<WIN>(p, idx);
    const int rows = u.rows_s[slot];
    if (rows <= 0) continue;
    const int t = 2 * u.pair + slot;
    const bool row_ok = r < rows;
    const int64_t grow = static_cast<int64_t>(u.seg.q0) + t * kTile + r;
    __nv_bfloat16* out_row = p.out + (grow * H + u.h) * D;
    const int nkv = u.nkv_s[slot];
    if (nkv == 0) {  // no keys: O = 0, LSE = -inf
      if (row_ok) {
#pragma unroll
        for (int c = 0; c < D; c += 8) st_global_v4(out_row + c, 0u, 0u, 0u, 0u);
        if (kSoftmax && p.lse) p.lse[static_cast<int64_t>(u.h) * p.total_q + grow] = -INFINITY;
      }
      continue;
    }
    float m_run = -INFINITY, l_run = 0.f;  // softmax state (base 2)
    float bc_lo = 0.f, bc_hi = 0.f;
    if (p.bias_len) {
      const float* brow = p.bias + static_cast<int64_t>(u.h) * p.bias_len;
      bc_lo = __ldg(brow);
      bc_hi = __ldg(brow + p.bias_len - 1);
    }
    bool ok = true;
    const int kfirst = u.k0 + u.beg_s[slot];  // this slot's key/value tiles: kfirst .. kend - 1
    const int kend = kfirst + nkv;
    for (int kt = kfirst; kt < kend; ++kt) {
      if (!(ok = mbar_wait(&bars->s_full[slot], s_it & 1, fail))) break;
      ++s_it;
      tc_fence_after();
      const int j0 = kt * kTile;
      const int i_row = t * kTile + r;  // segment-local query row
      // valid columns of this row: lo <= c < nvalid
      int nvalid = min(kTile, u.seg.lkv - j0);
      if (p.causal) nvalid = min(nvalid, i_row - j0 + 1);
      int lo = 0;
      bool tile_masked = (u.seg.lkv - j0 < kTile) || (p.causal && kt == t);
      if constexpr (WIN) {  // j0 + c in (i - w, i + w); each bound is formed only where it binds
        const int dj = i_row - j0;
        if (p.window <= kTile - dj) nvalid = min(nvalid, dj + p.window);
        if (dj >= p.window) lo = dj - p.window + 1;
        tile_masked = tile_masked || abs(t - kt) * kTile + (kTile - 1) >= p.window;
      }
      const int nchunks = (min(kTile, u.seg.lkv - j0) + 31) / 32;
      const TileBias tb = tile_bias(p, u.h, t * kTile, r, j0, bc_lo, bc_hi);
      if constexpr (!kSoftmax) {
        const float hs = 0.5f * p.scale;
        if (tb.band) {
          if (tile_masked) tile_act<ACT, NALU, true, true>(t_s, hs, tb, lo, nvalid, nchunks);
          else tile_act<ACT, NALU, true, false>(t_s, hs, tb, lo, nvalid, nchunks);
        } else {
          if (tile_masked) tile_act<ACT, NALU, false, true>(t_s, hs, tb, lo, nvalid, nchunks);
          else tile_act<ACT, NALU, false, false>(t_s, hs, tb, lo, nvalid, nchunks);
        }
      } else {
        const bool first = kt == kfirst;
        if (tb.band) {
          if (tile_masked) tile_softmax<D, true, true>(t_s, t_o, p.scale, tb, lo, nvalid, first, m_run, l_run);
          else tile_softmax<D, true, false>(t_s, t_o, p.scale, tb, lo, nvalid, first, m_run, l_run);
        } else {
          if (tile_masked) tile_softmax<D, false, true>(t_s, t_o, p.scale, tb, lo, nvalid, first, m_run, l_run);
          else tile_softmax<D, false, false>(t_s, t_o, p.scale, tb, lo, nvalid, first, m_run, l_run);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive_warp(&bars->p_full[slot]);
    }
    if (!ok) break;
    // epilogue: O (TMEM) -> bf16 -> global, rows < Lq only
    if (!mbar_wait(&bars->o_full[slot], o_it & 1, fail)) break;
    ++o_it;
    tc_fence_after();
    // softmax: a row that met no key (possible under a sliding window) has
    // l = 0 and O = 0; it keeps O = 0 and gets LSE = -inf
    const float inv_l = kSoftmax ? (l_run > 0.f ? 1.0f / l_run : 0.f) : 1.0f;
    if constexpr (FwdSmem<D, ACT>::kStage) {
      // A thread owns one row and rows lie H D 2 bytes apart, so plain stores
      // would touch 32 lines per instruction.  Each 64-column half of the
      // warp's 32 rows is staged in the warp's own 4 KB of shared memory
      // (XOR-swizzled 16-byte chunks), then stored four whole 128-byte rows
      // per instruction.
      // A block whose 32 rows all lie in the segment leaves by one TMA
      // store (the O map's 32-row box and 128-byte swizzle match the
      // staging); O is released once its last columns are in registers.
      const int lr = threadIdx.x & 31;
      uint8_t* stg_p = smem + C::kEpiOff + (warp - 4) * 4096;
      const uint32_t stg = smem_u32(stg_p);
      const int64_t row0 = grow - lr;  // global row of the warp's first row
      const bool whole = quad * 32 + 31 < rows;
#pragma unroll
      for (int hb = 0; hb < D / 64; ++hb) {
        if (lr == 0) bulk_wait_read_all();  // the staging's previous TMA store has read it
        __syncwarp();
#pragma unroll
        for (int c0 = 0; c0 < 64; c0 += 32) {
          uint32_t o[32];
          tmem_ld32(t_o + 64 * hb + c0, o);
          tmem_ld_wait(o);
          if (hb == D / 64 - 1 && c0 == 32) {
            tc_fence_before();
            mbar_arrive_warp(&bars->o_empty[slot]);
          }
#pragma unroll
          for (int c = 0; c < 32; c += 8) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
              w[e] = pack_bf16(__uint_as_float(o[c + 2 * e]) * inv_l, __uint_as_float(o[c + 2 * e + 1]) * inv_l);
            const int j = (c0 + c) >> 3;
            st_shared_v4(stg + lr * 128 + ((j ^ (lr & 7)) << 4), w[0], w[1], w[2], w[3]);
          }
        }
        if (whole) {
          fence_proxy_async_smem();
          __syncwarp();
          if (lr == 0) {
            tma_store_3d(&p.tm_o, stg_p, 64 * hb, u.h, static_cast<int>(row0));
            bulk_commit();
          }
        } else {
          __syncwarp();
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const int rr = 4 * k + (lr >> 3), j = lr & 7;
            uint32_t a, b2, c2, d2;
            ld_shared_v4(stg + rr * 128 + ((j ^ (rr & 7)) << 4), a, b2, c2, d2);
            if (quad * 32 + rr < rows)
              st_global_v4(p.out + ((row0 + rr) * H + u.h) * D + 64 * hb + 8 * j, a, b2, c2, d2);
          }
          __syncwarp();
        }
      }
    } else {
      // 32-byte stores where out allows them: half the store instructions,
      // whole 32-byte sectors (a thread owns one row, so each instruction
      // still touches 32 rows)
      const bool v8 = (reinterpret_cast<uintptr_t>(p.out) & 31) == 0;
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += 32) {
        uint32_t o[32];
        tmem_ld32(t_o + c0, o);
        tmem_ld_wait(o);
        if (row_ok) {
#pragma unroll
          for (int c = 0; c < 32; c += 16) {
            uint32_t w[8];
#pragma unroll
            for (int e = 0; e < 8; ++e)
              w[e] = pack_bf16(__uint_as_float(o[c + 2 * e]) * inv_l, __uint_as_float(o[c + 2 * e + 1]) * inv_l);
            if (v8) {
              st_global_v8(out_row + c0 + c, w);
            } else {
              st_global_v4(out_row + c0 + c, w[0], w[1], w[2], w[3]);
              st_global_v4(out_row + c0 + c + 8, w[4], w[5], w[6], w[7]);
            }
          }
        }
      }
    }
    if constexpr (!FwdSmem<D, ACT>::kStage) {
      tc_fence_before();
      mbar_arrive_warp(&bars->o_empty[slot]);
    }
    if (kSoftmax && row_ok && p.lse)
      p.lse[static_cast<int64_t>(u.h) * p.total_q + grow] = l_run > 0.f ? (m_run + __log2f(l_run)) * kLn2 : -INFINITY;
  }
  if constexpr (FwdSmem<D, ACT>::kStage) {  // this warp's TMA stores are complete before the CTA exits
    if ((threadIdx.x & 31) == 0) bulk_wait_all();
    __syncwarp();
  }
}

// ----------------------------------------------------------------- kernel
template <int D, int ACT, int NALU, bool WIN>
__global__ void __launch_bounds__(384, 1) gdpa_fwd_kernel(const __grid_constant__ FwdParams p) {
  using C = FwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  FwdBars* bars = reinterpret_cast<FwdBars*>(smem + FwdSmem<D, ACT>::kBarOff);
  const int warp = threadIdx.x >> 5;

  if (threadIdx.x == 0) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars->q_full[s], 1);
      mbar_init(&bars->q_empty[s], 1);
      mbar_init(&bars->s_full[s], 1);
      mbar_init(&bars->p_full[s], 4);
      mbar_init(&bars->o_full[s], 1);
      mbar_init(&bars->o_empty[s], 4);
    }
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&bars->k_full[s], 1);
      mbar_init(&bars->k_empty[s], 1);
      mbar_init(&bars->v_full[s], 1);
      mbar_init(&bars->v_empty[s], 1);
    }
    mbar_init(&bars->drain, 1);
    bars->abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&bars->tmem_base, C::kTmemCols);
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
    fwd_producer<D, WIN>(p, smem, bars, n_units, fail);
  } else if (warp == 1) {
    fwd_mma<D, WIN>(p, smem, bars, tmem, n_units, fail);
  } else if (warp >= 4) {
    fwd_act<D, ACT, NALU, WIN>(p, smem, bars, tmem, (warp - 4) >> 2, n_units, fail);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, C::kTmemCols);
}

// ======================================= forward, key/value tile resident
// For segments whose keys fit one tile (short key/value streams, e.g.
// cross-attention to a few memory tokens): every query tile meets the same
// single key/value tile.  The general kernel pairs two query tiles per unit
// and reloads that tile for each pair, and its next unit's loads wait for the
// current unit's products, so on such segments the load latency sets the
// pace.  Here a unit is (segment, head, chunk of up to kChunkTiles query
// tiles): K and V are loaded once per unit (two sets, so the next unit's pair
// loads while this one runs) and the query tiles stream through a ring,
// released as soon as their S product has read them.  The CTA's n-th query
// tile goes to activation warpgroup n % 2 (TMEM S_w, O_w), so one
// warpgroup's epilogue overlaps the other's activation.  P V is complete
// after one product, and softmax needs no running rescale.
// (The outer-loop pipelining of short inner loops: "Meta redesigns AI
// training infrastructure ...", section "Custom Kernels and 5D Parallelism
// ...".)
template <int D>
struct KvrCfg {
  using F = FwdCfg<D>;
  static constexpr int kQStages = D == 128 ? 2 : 4;
  static constexpr int kKvOff = 0;  // (K, V) set s: K at s 2 tiles, V one tile after
  static constexpr int kQOff = kKvOff + 4 * F::kTileBytes;
  static constexpr int kEpiOff = kQOff + kQStages * F::kTileBytes;
};
template <int D, int ACT>
struct KvrSmem {
  static constexpr bool kStage = D >= 64 && ACT != 2;
  static constexpr int kBarOff = KvrCfg<D>::kEpiOff + (kStage ? 8 * 4096 : 0);
  static constexpr int kSmemBytes = kBarOff + 512 + 1024;
  static_assert(kSmemBytes <= 232448, "shared memory per CTA");
};

struct KvrBars {
  uint64_t kv_full[2], kv_empty[2];
  uint64_t q_full[4], q_empty[4];
  uint64_t s_full[2], p_full[2], o_full[2], o_empty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};

// Query tiles [t0, t0 + nt) of segment b, head h.
struct KvrUnit {
  int b, h;
  Seg seg;
  int t0, nt;
};

__device__ __forceinline__ KvrUnit kvr_unit(const FwdParams& p, int idx) {
  KvrUnit u;
  const Unit w = p.units[idx];
  u.b = w.x;
  u.h = w.y;
  u.seg = load_seg(p.q_off, p.kv_off, u.b);
  u.t0 = w.z * kChunkTiles;
  u.nt = max(0, min(ceil_div(u.seg.lq, kTile) - u.t0, kChunkTiles));
  return u;
}

template <int D>
__device__ void kvr_producer(const FwdParams& p, uint8_t* smem, KvrBars* bars, int n_units, Fail fail) {
  using F = FwdCfg<D>;
  using C = KvrCfg<D>;
  uint32_t u_it = 0, q_it = 0;
  const bool leader = elect_one();
  bool ok = true;
  for (int r = 0; ok; ++r) {
    const int idx = unit_index(r, blockIdx.x, gridDim.x);
    if (idx >= n_units) break;
    const KvrUnit u = kvr_unit(p, idx);
    if (u.nt == 0) continue;
    const int ks = u_it & 1;
    if (!(ok = mbar_wait_warp(&bars->kv_empty[ks], ((u_it >> 1) & 1) ^ 1, fail))) break;
    if (leader) {
      mbar_arrive_tx(&bars->kv_full[ks], 2 * F::kTileBytes);
      uint8_t* kd = smem + C::kKvOff + ks * 2 * F::kTileBytes;
#pragma unroll
      for (int cb = 0; cb < F::kNumBlocks; ++cb) {
        tma_load_3d(kd + cb * F::kBlockBytes, &p.tm_k, &bars->kv_full[ks], cb * F::kBlockCols, u.h, u.seg.k0);
        tma_load_3d(kd + F::kTileBytes + cb * F::kBlockBytes, &p.tm_v, &bars->kv_full[ks], cb * F::kBlockCols, u.h,
                    u.seg.k0);
      }
    }
    ++u_it;
    // shared queries: the Q map holds the shared rows once
    const int qrow0 = p.q_shared ? 0 : u.seg.q0;
    for (int t = 0; t < u.nt && ok; ++t) {
      const int st = q_it % C::kQStages;
      if (!(ok = mbar_wait_warp(&bars->q_empty[st], ((q_it / C::kQStages) & 1) ^ 1, fail))) break;
      if (leader) {
        mbar_arrive_tx(&bars->q_full[st], F::kTileBytes);
        uint8_t* qd = smem + C::kQOff + st * F::kTileBytes;
#pragma unroll
        for (int cb = 0; cb < F::kNumBlocks; ++cb)
          tma_load_3d(qd + cb * F::kBlockBytes, &p.tm_q, &bars->q_full[st], cb * F::kBlockCols, u.h,
                      qrow0 + (u.t0 + t) * kTile);
      }
      ++q_it;
    }
  }
  if (!ok) {  // let the copies already issued land before the CTA exits
    for (uint32_t i = u_it > 2 ? u_it - 2 : 0; i < u_it; ++i) mbar_wait_drain(&bars->kv_full[i & 1], (i >> 1) & 1);
    for (uint32_t i = q_it > C::kQStages ? q_it - C::kQStages : 0; i < q_it; ++i)
      mbar_wait_drain(&bars->q_full[i % C::kQStages], (i / C::kQStages) & 1);
  }
}

template <int D>
__device__ void kvr_mma(const FwdParams& p, uint8_t* smem, KvrBars* bars, uint32_t tmem, int n_units, Fail fail) {
  using F = FwdCfg<D>;
  using C = KvrCfg<D>;
  uint32_t u_it = 0, n = 0;
  const bool leader = elect_one();
  bool ok = true;
  for (int r = 0; ok; ++r) {
    const int idx = unit_index(r, blockIdx.x, gridDim.x);
    if (idx >= n_units) break;
    const KvrUnit u = kvr_unit(p, idx);
    if (u.nt == 0) continue;
    const int ks = u_it & 1;
    if (!(ok = mbar_wait_warp(&bars->kv_full[ks], (u_it >> 1) & 1, fail))) break;
    ++u_it;
    const uint32_t k_addr = smem_u32(smem + C::kKvOff + ks * 2 * F::kTileBytes);
    const uint32_t v_addr = k_addr + F::kTileBytes;
    // S of tile m into S_(m % 2): the columns that P V of tile m - 2 read,
    // issued before it (MMAs execute in issue order)
    auto issue_s = [&](uint32_t m) -> bool {
      const int st = m % C::kQStages, w = m & 1;
      if (!mbar_wait_warp(&bars->q_full[st], (m / C::kQStages) & 1, fail)) return false;
      tc_fence_after();
      issue_qk<D>(tmem + 128 * w, smem_u32(smem + C::kQOff + st * F::kTileBytes), k_addr, leader);
      if (leader) mma_commit(&bars->s_full[w]);
      if (leader) mma_commit(&bars->q_empty[st]);  // the query tile is read by S only
      return true;
    };
    if (!(ok = issue_s(n))) break;
    for (int t = 0; t < u.nt && ok; ++t) {
      const uint32_t m = n + t;
      const int w = m & 1;
      if (t + 1 < u.nt && !(ok = issue_s(m + 1))) break;
      if (!(ok = mbar_wait_warp(&bars->o_empty[w], ((m >> 1) & 1) ^ 1, fail))) break;
      if (!(ok = mbar_wait_warp(&bars->p_full[w], (m >> 1) & 1, fail))) break;
      tc_fence_after();
      issue_pv<D>(tmem + 256 + D * w, tmem + 128 * w, v_addr, false, leader);
      if (leader) mma_commit(&bars->o_full[w]);
    }
    if (!ok) break;
    n += u.nt;
    if (leader) mma_commit(&bars->kv_empty[ks]);  // every product of this unit issued
  }
  if (leader) mma_commit(&bars->drain);
  mbar_wait_drain(&bars->drain, 0);
}

template <int D, int ACT>
__device__ void kvr_act(const FwdParams& p, uint8_t* smem, KvrBars* bars, uint32_t tmem, int w, int n_units,
                        Fail fail) {
  using C = KvrCfg<D>;
  constexpr bool kSoftmax = ACT == 2;
  const int warp = threadIdx.x >> 5;
  const int quad = warp & 3;
  const int r = quad * 32 + (threadIdx.x & 31);  // query row of the tile owned by this thread
  const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
  const uint32_t t_s = tmem + lane_off + 128 * w;
  const uint32_t t_o = tmem + lane_off + 256 + D * w;
  const int H = p.heads;
  uint32_t n = 0;
  for (int rr = 0;; ++rr) {
    const int idx = unit_index(rr, blockIdx.x, gridDim.x);
    if (idx >= n_units) break;
    const KvrUnit u = kvr_unit(p, idx);
    if (u.nt == 0) continue;
    float bc_lo = 0.f, bc_hi = 0.f;
    if (p.bias_len) {
      const float* brow = p.bias + static_cast<int64_t>(u.h) * p.bias_len;
      bc_lo = __ldg(brow);
      bc_hi = __ldg(brow + p.bias_len - 1);
    }
    const int nchunks = (min(kTile, u.seg.lkv) + 31) / 32;
    bool ok = true;
    for (int t = 0; t < u.nt; ++t) {
      const uint32_t m = n + t;
      if (static_cast<int>(m & 1) != w) continue;
      const int qt = u.t0 + t;
      const int rows = u.seg.lq - qt * kTile;
      if (!(ok = mbar_wait(&bars->s_full[w], (m >> 1) & 1, fail))) break;
      tc_fence_after();
      const int i_row = qt * kTile + r;  // segment-local query row
      int nvalid = min(kTile, u.seg.lkv);
      if (p.causal) nvalid = min(nvalid, i_row + 1);
      const bool tile_masked = u.seg.lkv < kTile || (p.causal && qt == 0);
      const TileBias tb = tile_bias(p, u.h, qt * kTile, r, 0, bc_lo, bc_hi);
      float m_run = -INFINITY, l_run = 0.f;  // softmax state (base 2)
      if constexpr (!kSoftmax) {
        const float hs = 0.5f * p.scale;
        if (tb.band) {
          if (tile_masked) tile_act<ACT, kFwdAluChunks, true, true>(t_s, hs, tb, 0, nvalid, nchunks);
          else tile_act<ACT, kFwdAluChunks, true, false>(t_s, hs, tb, 0, nvalid, nchunks);
        } else {
          if (tile_masked) tile_act<ACT, kFwdAluChunks, false, true>(t_s, hs, tb, 0, nvalid, nchunks);
          else tile_act<ACT, kFwdAluChunks, false, false>(t_s, hs, tb, 0, nvalid, nchunks);
        }
      } else {
        if (tb.band) {
          if (tile_masked) tile_softmax<D, true, true>(t_s, t_o, p.scale, tb, 0, nvalid, true, m_run, l_run);
          else tile_softmax<D, true, false>(t_s, t_o, p.scale, tb, 0, nvalid, true, m_run, l_run);
        } else {
          if (tile_masked) tile_softmax<D, false, true>(t_s, t_o, p.scale, tb, 0, nvalid, true, m_run, l_run);
          else tile_softmax<D, false, false>(t_s, t_o, p.scale, tb, 0, nvalid, true, m_run, l_run);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive_warp(&bars->p_full[w]);
      // epilogue: O (TMEM) -> bf16 -> global, rows < Lq only
      if (!(ok = mbar_wait(&bars->o_full[w], (m >> 1) & 1, fail))) break;
      tc_fence_after();
      const int64_t grow = static_cast<int64_t>(u.seg.q0) + qt * kTile + r;
      const float inv_l = kSoftmax ? (l_run > 0.f ? 1.0f / l_run : 0.f) : 1.0f;
      if constexpr (KvrSmem<D, ACT>::kStage) {
        // each 64-column half of the warp's 32 rows staged in the warp's own
        // 4 KB (the 128-byte swizzle of the O tensor map); a block whose 32
        // rows all lie in the segment leaves by one TMA store, the last
        // block of a segment by stores of four whole 128-byte rows per
        // instruction
        const int lr = threadIdx.x & 31;
        uint8_t* stg_p = smem + C::kEpiOff + (warp - 4) * 4096;
        const uint32_t stg = smem_u32(stg_p);
        const int64_t row0 = grow - lr;
        const bool whole = quad * 32 + 31 < rows;
#pragma unroll
        for (int hb = 0; hb < D / 64; ++hb) {
          if (lr == 0) bulk_wait_read_all();  // the block's previous TMA store has read it
          __syncwarp();
#pragma unroll
          for (int c0 = 0; c0 < 64; c0 += 32) {
            uint32_t o[32];
            tmem_ld32(t_o + 64 * hb + c0, o);
            tmem_ld_wait(o);
            if (hb == D / 64 - 1 && c0 == 32) {  // every column of O is in registers
              tc_fence_before();
              mbar_arrive_warp(&bars->o_empty[w]);
            }
#pragma unroll
            for (int c = 0; c < 32; c += 8) {
              uint32_t wd[4];
#pragma unroll
              for (int e = 0; e < 4; ++e)
                wd[e] = pack_bf16(__uint_as_float(o[c + 2 * e]) * inv_l, __uint_as_float(o[c + 2 * e + 1]) * inv_l);
              const int j = (c0 + c) >> 3;
              st_shared_v4(stg + lr * 128 + ((j ^ (lr & 7)) << 4), wd[0], wd[1], wd[2], wd[3]);
            }
          }
          if (whole) {
            fence_proxy_async_smem();
            __syncwarp();
            if (lr == 0) {
              tma_store_3d(&p.tm_o, stg_p, 64 * hb, u.h, static_cast<int>(row0));
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
                st_global_v4(p.out + ((row0 + rw) * H + u.h) * D + 64 * hb + 8 * j, a, b2, c2, d2);
            }
            __syncwarp();
          }
        }
      } else {
        __nv_bfloat16* out_row = p.out + (grow * H + u.h) * D;
        const bool v8 = (reinterpret_cast<uintptr_t>(p.out) & 31) == 0;
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += 32) {
          uint32_t o[32];
          tmem_ld32(t_o + c0, o);
          tmem_ld_wait(o);
          if (c0 + 32 == D) {
            tc_fence_before();
            mbar_arrive_warp(&bars->o_empty[w]);
          }
          if (r < rows) {  // 32-byte stores where out allows them (as in the general kernel)
#pragma unroll
            for (int c = 0; c < 32; c += 16) {
              uint32_t wd[8];
#pragma unroll
              for (int e = 0; e < 8; ++e)
                wd[e] = pack_bf16(__uint_as_float(o[c + 2 * e]) * inv_l, __uint_as_float(o[c + 2 * e + 1]) * inv_l);
              if (v8) {
                st_global_v8(out_row + c0 + c, wd);
              } else {
                st_global_v4(out_row + c0 + c, wd[0], wd[1], wd[2], wd[3]);
                st_global_v4(out_row + c0 + c + 8, wd[4], wd[5], wd[6], wd[7]);
              }
            }
          }
        }
      }
      if (kSoftmax && r < rows && p.lse)
        p.lse[static_cast<int64_t>(u.h) * p.total_q + grow] = l_run > 0.f ? (m_run + __log2f(l_run)) * kLn2 : -INFINITY;
    }
    if (!ok) break;
    n += u.nt;
  }
  if constexpr (KvrSmem<D, ACT>::kStage) {  // this warp's TMA stores are complete before the CTA exits
    if ((threadIdx.x & 31) == 0) bulk_wait_all();
    __syncwarp();
  }
}

template <int D, int ACT>
__global__ void __launch_bounds__(384, 1) gdpa_fwd_kvres_kernel(const __grid_constant__ FwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  KvrBars* bars = reinterpret_cast<KvrBars*>(smem + KvrSmem<D, ACT>::kBarOff);
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars->kv_full[s], 1);
      mbar_init(&bars->kv_empty[s], 1);
      mbar_init(&bars->s_full[s], 1);
      mbar_init(&bars->p_full[s], 4);
      mbar_init(&bars->o_full[s], 1);
      mbar_init(&bars->o_empty[s], 4);
    }
    for (int s = 0; s < 4; ++s) {
      mbar_init(&bars->q_full[s], 1);
      mbar_init(&bars->q_empty[s], 1);
    }
    mbar_init(&bars->drain, 1);
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
  if (warp == 0) kvr_producer<D>(p, smem, bars, n_units, fail);
  else if (warp == 1) kvr_mma<D>(p, smem, bars, tmem, n_units, fail);
  else if (warp >= 4) kvr_act<D, ACT>(p, smem, bars, tmem, (warp - 4) >> 2, n_units, fail);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

// ------------------------------------------------------------------ launch
// Each object file holds the kernels of one head dimension (JGDPA_HEAD_DIM),
// so that the build compiles the head dimensions in parallel.
#ifndef JGDPA_HEAD_DIM
#error "compile fwd.cu with -DJGDPA_HEAD_DIM=32, 64 or 128"
#endif

template <int D, int ACT>
static cudaError_t launch_fwd_t(const FwdParams& p, int grid, cudaStream_t stream) {
  auto kern = p.window > 0 ? gdpa_fwd_kernel<D, ACT, kFwdAluChunks, true> : gdpa_fwd_kernel<D, ACT, kFwdAluChunks, false>;
  constexpr int kSmemBytes = FwdSmem<D, ACT>::kSmemBytes;
  static DeviceFlags attr_set[2] = {};
  cudaError_t e = smem_attr_once(kern, kSmemBytes, attr_set[p.window > 0]);
  if (e != cudaSuccess) return e;
  kern<<<grid, 384, kSmemBytes, stream>>>(p);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_fwd_d(const FwdParams& p, int act, int grid, cudaStream_t stream) {
  if (act == 0) return launch_fwd_t<D, 0>(p, grid, stream);
  if (act == 1) return launch_fwd_t<D, 1>(p, grid, stream);
  return launch_fwd_t<D, 2>(p, grid, stream);
}
template cudaError_t launch_fwd_d<JGDPA_HEAD_DIM>(const FwdParams&, int, int, cudaStream_t);

// The key/value-resident forward (segments whose keys fit one tile; no window).
template <int ACT>
static cudaError_t launch_kvres_t(const FwdParams& p, int grid, cudaStream_t stream) {
  constexpr int D = JGDPA_HEAD_DIM;
  auto kern = gdpa_fwd_kvres_kernel<D, ACT>;
  // at least half the SM's shared memory: one CTA per SM, so that a second
  // CTA never waits in its TMEM allocation for the first to finish
  constexpr int kSmem = KvrSmem<D, ACT>::kSmemBytes > 120 * 1024 ? KvrSmem<D, ACT>::kSmemBytes : 120 * 1024;
  static DeviceFlags attr_set = {};
  cudaError_t e = smem_attr_once(kern, kSmem, attr_set);
  if (e != cudaSuccess) return e;
  kern<<<grid, 384, kSmem, stream>>>(p);
  return cudaGetLastError();
}
template <int D>
cudaError_t launch_fwd_kvres_d(const FwdParams& p, int act, int grid, cudaStream_t stream) {
  if (act == 0) return launch_kvres_t<0>(p, grid, stream);
  if (act == 1) return launch_kvres_t<1>(p, grid, stream);
  return launch_kvres_t<2>(p, grid, stream);
}
template cudaError_t launch_fwd_kvres_d<JGDPA_HEAD_DIM>(const FwdParams&, int, int, cudaStream_t);

}  // namespace jg
