// Short-query backward for sm_103a: every segment reads the same NQ <= 64
// shared query rows (PMA-style pooling: "GEM Training: How Meta Doubled the
// Efficiency of Its ..." (globalainews.in), section "What to watch").
//
// The keys take the MMA's 128 rows and the queries are N (swap-AB), so the
// activation and the tiles touch only the NQ live query columns:
//   S^T = K Q^T, dP^T = V dO^T            128 keys x NQ, fp32 in TMEM
//   P^T = act(x)^T, dS^T = (dP act'(x))^T  activation warps; bf16 back into
//                                          TMEM over S^T and dP^T, and dS
//                                          into a shared [NQ][128 keys] tile
//   dV = P^T dO, dK = s dS^T Q            A operand from TMEM, K = NQ
//   dQ^T += K^T dS^T                       M = 128 rows of d, N = NQ
// With at most NQ query rows every key tile is finished after one such step:
// dK and dV are written per tile, and no dS is stored.  A unit is (segment,
// head, chunk of up to kChunkTiles key tiles); its dQ contribution
// accumulates in TMEM over the chunk and is written once, in fp32, to the
// unit's own block; a fixed-order reduction sums the blocks (the split dQ
// without atomics of "Meta redesigns AI training infrastructure ...",
// section "Eliminating Compute Waste in Asymmetric Workloads").
//
// Warp roles (384 threads):
//   warp 0      TMA producer: the unit's Q and dO blocks, K / V tiles into rings
//   warp 1      MMA issuer; owns TMEM
//   warps 4-7   activation: one key row per thread
//   warps 8-11  epilogue: dV, dK per tile (TMEM -> bf16 -> global), the
//               unit's dQ contribution (TMEM lane = column of d)
// GELU / SiLU (softmax goes to the general backward).
#include "act.cuh"
#include "common.cuh"
#include "ptx.cuh"

namespace jg {

template <int D, int NQ>
struct BsqCfg {
  static constexpr int kBlockCols = D < 64 ? D : 64;
  static constexpr int kRowBytes = kBlockCols * 2;
  static constexpr int kNumBlocks = D / kBlockCols;
  static constexpr uint32_t kSwizzle = kRowBytes == 128 ? 2u : 4u;
  static constexpr int kSBO = 8 * kRowBytes;
  static constexpr int kTileBlockBytes = kTile * kRowBytes;  // one column block of a 128-row tile
  static constexpr int kTileBytes = kTile * D * 2;
  static constexpr int kQBlockBytes = NQ * kRowBytes;        // one column block of an NQ-row block
  static constexpr int kQBytes = NQ * D * 2;
  static constexpr int kDsBlockBytes = NQ * 128;             // 64 keys of the dS tile
  static constexpr int kDsBytes = NQ * kTile * 2;
  // TMEM columns: S^T and dP^T (double-buffered where they fit), dV, dK, dQ^T
  static constexpr int kNumBuf = 5 * NQ + 2 * D <= 512 ? 2 : 1;
  static constexpr int kColS = 0;
  static constexpr int kColDp = kNumBuf * NQ;
  static constexpr int kColDv = 2 * kNumBuf * NQ;
  static constexpr int kColDk = kColDv + D;
  static constexpr int kColDq = kColDk + D;
  static_assert(kColDq + NQ <= 512, "TMEM columns");
  // Shared memory: the K ring, then the V ring (for d < 128 the K^T operand
  // of dQ^T spans 128 rows of d, and its rows >= d read the memory after the
  // K tile, which this order keeps inside the allocation: see bsq_mma_dq),
  // Q, dO, two dS tiles, the epilogue's per-warp staging, barriers.
  static constexpr int kStages = D == 128 ? (NQ == 16 ? 3 : 2) : 4;
  static constexpr int kKOff = 0;
  static constexpr int kVOff = kKOff + kStages * kTileBytes;
  static constexpr int kQOff = kVOff + kStages * kTileBytes;
  static constexpr int kDoOff = kQOff + kQBytes;
  static constexpr int kDsOff = kDoOff + kQBytes;
  static constexpr int kStageOff = kDsOff + 2 * kDsBytes;
  static constexpr int kBarOff = kStageOff + (D >= 64 ? 4 * 4096 : 0);
  static constexpr int kSmemBytes = kBarOff + 512 + 1024;
  static_assert(kSmemBytes <= 232448, "shared memory per CTA");
  static_assert(kKOff + (kStages - 1) * kTileBytes + (kTile / kBlockCols) * kTileBlockBytes <= kQOff,
                "K^T operand rows stay inside the K and V rings");
};

struct BsqBars {
  uint64_t qd_full, qd_empty;
  uint64_t kv_full[4], kv_empty[4];
  uint64_t s_full[2];               // S^T, dP^T of a tile in TMEM (MMA -> activation)
  uint64_t pds_full[2];             // P^T, dS^T in TMEM and dS in shared memory (activation -> MMA)
  uint64_t ds_empty[2];             // a dS tile read by its dQ^T MMA
  uint64_t acc_full, acc_empty;     // dV, dK of a tile (MMA <-> epilogue)
  uint64_t dq_full, dq_empty;       // the unit's dQ^T (MMA <-> epilogue)
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};

// Key tiles [t0, t0 + nt) of segment b, head h.
struct BsqUnit {
  int b, h, chunk;
  Seg seg;
  int t0, nt;
};

__device__ __forceinline__ BsqUnit bsq_unit(const BwdParams& p, int idx) {
  BsqUnit u;
  const Unit w = p.units[idx];
  u.b = w.x;
  u.h = w.y;
  u.chunk = w.z;
  u.seg = load_seg(p.q_off, p.kv_off, u.b);
  u.t0 = u.chunk * kChunkTiles;
  u.nt = max(0, min(ceil_div(u.seg.lkv, kTile) - u.t0, kChunkTiles));
  return u;
}

// ------------------------------------------------------------- producer
template <int D, int NQ>
__device__ void bsq_producer(const BwdParams& p, uint8_t* smem, BsqBars* bars, int n_units, Fail fail) {
  using C = BsqCfg<D, NQ>;
  uint32_t u_it = 0, kv_it = 0;
  const bool leader = elect_one();
  bool ok = true;
  for (int r = 0; ok; ++r) {
    const int idx = unit_index(r, blockIdx.x, gridDim.x);
    if (idx >= n_units) break;
    const BsqUnit u = bsq_unit(p, idx);
    if (u.nt == 0) continue;
    if (!(ok = mbar_wait_warp(&bars->qd_empty, (u_it & 1) ^ 1, fail))) break;
    if (leader) {  // the shared query block (row 0) and this segment's dO rows
      mbar_arrive_tx(&bars->qd_full, 2 * C::kQBytes);
#pragma unroll
      for (int cb = 0; cb < C::kNumBlocks; ++cb) {
        tma_load_3d(smem + C::kQOff + cb * C::kQBlockBytes, &p.tm_q, &bars->qd_full, cb * C::kBlockCols, u.h, 0);
        tma_load_3d(smem + C::kDoOff + cb * C::kQBlockBytes, &p.tm_do, &bars->qd_full, cb * C::kBlockCols, u.h,
                    u.seg.q0);
      }
    }
    ++u_it;
    for (int t = 0; t < u.nt && ok; ++t) {
      const int st = kv_it % C::kStages;
      const int row = u.seg.k0 + (u.t0 + t) * kTile;
      if (!(ok = mbar_wait_warp(&bars->kv_empty[st], ((kv_it / C::kStages) & 1) ^ 1, fail))) break;
      if (leader) {
        mbar_arrive_tx(&bars->kv_full[st], 2 * C::kTileBytes);
#pragma unroll
        for (int cb = 0; cb < C::kNumBlocks; ++cb) {
          tma_load_3d(smem + C::kKOff + st * C::kTileBytes + cb * C::kTileBlockBytes, &p.tm_k, &bars->kv_full[st],
                      cb * C::kBlockCols, u.h, row);
          tma_load_3d(smem + C::kVOff + st * C::kTileBytes + cb * C::kTileBlockBytes, &p.tm_v, &bars->kv_full[st],
                      cb * C::kBlockCols, u.h, row);
        }
      }
      ++kv_it;
    }
  }
  if (!ok) {  // let the copies already issued land before the CTA exits
    if (u_it) mbar_wait_drain(&bars->qd_full, (u_it - 1) & 1);
    for (uint32_t i = kv_it > C::kStages ? kv_it - C::kStages : 0; i < kv_it; ++i)
      mbar_wait_drain(&bars->kv_full[i % C::kStages], (i / C::kStages) & 1);
  }
}

// ------------------------------------------------------------ MMA issuer
// C(tmem, 128 keys x NQ) = T (128 x D, K-major) * U (NQ x D, K-major)^T:
// S^T with (K, Q), dP^T with (V, dO).
template <int D, int NQ>
__device__ __forceinline__ void bsq_mma_t(uint32_t d_tmem, uint32_t t_tile, uint32_t u_blk, bool leader) {
  using C = BsqCfg<D, NQ>;
  constexpr uint32_t idesc = idesc_bf16(kTile, NQ, 0, 0);
  const uint64_t a0 = sdesc(t_tile, 16, C::kSBO, C::kSwizzle), b0 = sdesc(u_blk, 16, C::kSBO, C::kSwizzle);
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const int blk = kk * 16 / C::kBlockCols, col2 = (kk * 16 % C::kBlockCols) * 2;
    const uint64_t aoff = static_cast<uint64_t>(blk * C::kTileBlockBytes + col2) >> 4;
    const uint64_t boff = static_cast<uint64_t>(blk * C::kQBlockBytes + col2) >> 4;
    if (leader) mma_ss(d_tmem, a0 + aoff, b0 + boff, idesc, kk > 0 ? 1u : 0u);
  }
}
// C(tmem, 128 keys x D) = A (TMEM, 128 keys x NQ bf16) * U (NQ x D, MN-major):
// dV with (P^T, dO), dK with (dS^T, Q).
template <int D, int NQ>
__device__ __forceinline__ void bsq_mma_a_tmem(uint32_t d_tmem, uint32_t a_tmem, uint32_t u_blk, bool leader) {
  using C = BsqCfg<D, NQ>;
  constexpr uint32_t idesc = idesc_bf16(kTile, D, 0, 1);
  const uint64_t b0 = sdesc(u_blk, C::kQBlockBytes, C::kSBO, C::kSwizzle);
#pragma unroll
  for (int kk = 0; kk < NQ / 16; ++kk) {
    const uint64_t boff = static_cast<uint64_t>(kk * 16 * C::kRowBytes) >> 4;
    if (leader) mma_ts(d_tmem, a_tmem + kk * 8, b0 + boff, idesc, kk > 0 ? 1u : 0u);
  }
}
// dQ^T (tmem, 128 x NQ; lane = column of d) (+)= K^T (M = 128 along d, K =
// 128 keys: the K tile read as an MN-major operand) * dS^T (the dS tile
// [NQ][128 keys], K-major).  For d < 128 the rows d..127 of the operand are
// the memory after the K tile (the next ring slots): the matching TMEM lanes
// are never read.
template <int D, int NQ>
__device__ __forceinline__ void bsq_mma_dq(uint32_t d_tmem, uint32_t k_tile, uint32_t ds_tile, bool accumulate,
                                           bool leader) {
  using C = BsqCfg<D, NQ>;
  constexpr uint32_t idesc = idesc_bf16(kTile, NQ, 1, 0);
  const uint64_t a0 = sdesc(k_tile, C::kTileBlockBytes, C::kSBO, C::kSwizzle);
  const uint64_t b0 = sdesc(ds_tile, 16, 1024, 2u);
#pragma unroll
  for (int kk = 0; kk < kTile / 16; ++kk) {
    const uint64_t aoff = static_cast<uint64_t>(kk * 16 * C::kRowBytes) >> 4;
    const uint64_t boff = static_cast<uint64_t>((kk * 16 / 64) * C::kDsBlockBytes + (kk * 16 % 64) * 2) >> 4;
    if (leader) mma_ss(d_tmem, a0 + aoff, b0 + boff, idesc, (accumulate || kk > 0) ? 1u : 0u);
  }
}

template <int D, int NQ>
__device__ void bsq_mma(const BwdParams& p, uint8_t* smem, BsqBars* bars, uint32_t tmem, int n_units, Fail fail) {
  using C = BsqCfg<D, NQ>;
  const uint32_t k_base = smem_u32(smem + C::kKOff), v_base = smem_u32(smem + C::kVOff);
  const uint32_t q_blk = smem_u32(smem + C::kQOff), do_blk = smem_u32(smem + C::kDoOff);
  const uint32_t ds_base = smem_u32(smem + C::kDsOff);
  uint32_t u_it = 0, n = 0, acc_n = 0, dq_n = 0;
  const bool leader = elect_one();
  bool ok = true;
  // S^T and dP^T of tile m (ring slot m % stages) into TMEM buffer m % kNumBuf
  // (free: the dV / dK MMAs that read its P^T / dS^T were issued before)
  auto issue_sdp = [&](uint32_t m) -> bool {
    const int st = m % C::kStages, sb = m % C::kNumBuf;
    if (!mbar_wait_warp(&bars->kv_full[st], (m / C::kStages) & 1, fail)) return false;
    tc_fence_after();
    bsq_mma_t<D, NQ>(tmem + C::kColS + sb * NQ, k_base + st * C::kTileBytes, q_blk, leader);
    bsq_mma_t<D, NQ>(tmem + C::kColDp + sb * NQ, v_base + st * C::kTileBytes, do_blk, leader);
    if (leader) mma_commit(&bars->s_full[sb]);
    return true;
  };
  for (int r = 0; ok; ++r) {
    const int idx = unit_index(r, blockIdx.x, gridDim.x);
    if (idx >= n_units) break;
    const BsqUnit u = bsq_unit(p, idx);
    if (u.nt == 0) continue;
    if (!(ok = mbar_wait_warp(&bars->qd_full, u_it & 1, fail))) break;
    ++u_it;
    for (int t = 0; t < C::kNumBuf && t < u.nt && ok; ++t) ok = issue_sdp(n + t);
    for (int t = 0; t < u.nt && ok; ++t) {
      const uint32_t m = n + t;
      const int st = m % C::kStages, sb = m % C::kNumBuf, db = m & 1;
      if (!(ok = mbar_wait_warp(&bars->pds_full[db], (m >> 1) & 1, fail))) break;
      if (!(ok = mbar_wait_warp(&bars->acc_empty, (acc_n & 1) ^ 1, fail))) break;
      ++acc_n;
      tc_fence_after();
      bsq_mma_a_tmem<D, NQ>(tmem + C::kColDv, tmem + C::kColS + sb * NQ, do_blk, leader);  // dV = P^T dO
      bsq_mma_a_tmem<D, NQ>(tmem + C::kColDk, tmem + C::kColDp + sb * NQ, q_blk, leader);  // dK = dS^T Q
      if (leader) mma_commit(&bars->acc_full);
      if (t == 0) {  // the previous unit's dQ^T has been read
        if (!(ok = mbar_wait_warp(&bars->dq_empty, (dq_n & 1) ^ 1, fail))) break;
        ++dq_n;
        tc_fence_after();
      }
      bsq_mma_dq<D, NQ>(tmem + C::kColDq, k_base + st * C::kTileBytes, ds_base + db * C::kDsBytes, t > 0, leader);
      if (leader) mma_commit(&bars->ds_empty[db]);
      if (leader) mma_commit(&bars->kv_empty[st]);
      if (t + C::kNumBuf < u.nt) ok = issue_sdp(m + C::kNumBuf);
    }
    if (!ok) break;
    n += u.nt;
    if (leader) mma_commit(&bars->dq_full);
    if (leader) mma_commit(&bars->qd_empty);
  }
  if (leader) mma_commit(&bars->drain);
  mbar_wait_drain(&bars->drain, 0);
}

// ------------------------------------------------------ activation warps
// Byte offset of dS element (query row q, key c) in a dS tile: two 64-key
// column blocks of [NQ rows][128 bytes], 16-byte pieces swizzled by the row.
template <int NQ>
__device__ __forceinline__ uint32_t bsq_ds_offset(int q, int c) {
  return (c >> 6) * (NQ * 128) + q * 128 + ((((c & 63) >> 3) ^ (q & 7)) << 4) + (c & 7) * 2;
}

template <int D, int ACT, int NQ, bool WIN>
__device__ void bsq_act(const BwdParams& p, uint8_t* smem, BsqBars* bars, uint32_t tmem, int n_units, Fail fail) {
  using C = BsqCfg<D, NQ>;
  const int quad = (threadIdx.x >> 5) & 3;
  const int r = quad * 32 + (threadIdx.x & 31);  // key row of the tile (TMEM lane)
  const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
  const uint32_t ds_base = smem_u32(smem + C::kDsOff);
  const int H = p.heads;
  const int R = (p.bias_len - 1) / 2;
  const float hs = 0.5f * p.scale;  // x / 2 = hs S + bias / 2
  uint32_t n = 0;
  for (int rr = 0;; ++rr) {
    const int idx = unit_index(rr, blockIdx.x, gridDim.x);
    if (idx >= n_units) break;
    const BsqUnit u = bsq_unit(p, idx);
    if (u.nt == 0) continue;
    const float* brow = p.bias_len ? p.bias + static_cast<int64_t>(u.h) * p.bias_len : nullptr;
    unsigned long long* part =
        p.dbias_part ? p.dbias_part + (static_cast<int64_t>(blockIdx.x) * H + u.h) * p.bias_len : nullptr;
    const float bc_lo = brow ? __ldg(brow) : 0.f;
    float acc_lo = 0.f, acc_hi = 0.f;  // dbias mass clamped to the table's ends
    bool ok = true;
    for (int t = 0; t < u.nt; ++t, ++n) {
      const int sb = n % C::kNumBuf, db = n & 1;
      const int jt0 = (u.t0 + t) * kTile;  // first key of the tile
      const int j = jt0 + r;
      const bool j_ok = j < u.seg.lkv;
      // rel = q - j: some |rel| < R in this tile only while jt0 - (NQ - 1) < R;
      // otherwise every rel <= -R (the table's first entry)
      const bool band = brow != nullptr && jt0 - (NQ - 1) < R;
      if (!(ok = mbar_wait(&bars->s_full[sb], (n / C::kNumBuf) & 1, fail))) break;
      if (!(ok = mbar_wait(&bars->ds_empty[db], ((n >> 1) & 1) ^ 1, fail))) break;
      tc_fence_after();
      const uint32_t t_s = tmem + lane_off + C::kColS + sb * NQ;
      const uint32_t t_dp = tmem + lane_off + C::kColDp + sb * NQ;
      const uint32_t ds_tile = ds_base + db * C::kDsBytes;
#pragma unroll
      for (int c0 = 0; c0 < NQ; c0 += 16) {
        uint32_t sv[16], dv[16];
        tmem_ld16(t_s + c0, sv);
        tmem_ld16(t_dp + c0, dv);
        tmem_ld_wait16(sv);
        tmem_ld_wait16(dv);
        uint32_t ppk[8], dpk[8];
#pragma unroll
        for (int e2 = 0; e2 < 8; ++e2) {
          const int q = c0 + 2 * e2;  // query rows q, q + 1 (column of S^T)
          float2 bias = f2(bc_lo);
          if (band)
            bias = make_float2(ld_nc_f32(brow + min(max(q - j, -R), R) + R),
                               ld_nc_f32(brow + min(max(q + 1 - j, -R), R) + R));
          const float2 hx = __ffma2_rn(make_float2(__uint_as_float(sv[2 * e2]), __uint_as_float(sv[2 * e2 + 1])),
                                       f2(hs), __fmul2_rn(bias, f2(0.5f)));
          float2 kv;
          float2 pv = act2_d<ACT, false>(hx, kv);
          bool ok0 = j_ok && q < p.q_rows, ok1 = j_ok && q + 1 < p.q_rows;
          if (p.causal) {
            ok0 = ok0 && j <= q;
            ok1 = ok1 && j <= q + 1;
          }
          if constexpr (WIN) {
            ok0 = ok0 && abs(q - j) < p.window;
            ok1 = ok1 && abs(q + 1 - j) < p.window;
          }
          if (!ok0) pv.x = kv.x = 0.f;
          if (!ok1) pv.y = kv.y = 0.f;
          const float2 ds = __fmul2_rn(make_float2(__uint_as_float(dv[2 * e2]), __uint_as_float(dv[2 * e2 + 1])), kv);
          ppk[e2] = pack_bf16(pv.x, pv.y);
          dpk[e2] = pack_bf16(ds.x, ds.y);
          asm volatile("st.shared.u16 [%0], %1;" ::"r"(ds_tile + bsq_ds_offset<NQ>(q, r)),
                       "h"(static_cast<uint16_t>(dpk[e2] & 0xFFFFu))
                       : "memory");
          asm volatile("st.shared.u16 [%0], %1;" ::"r"(ds_tile + bsq_ds_offset<NQ>(q + 1, r)),
                       "h"(static_cast<uint16_t>(dpk[e2] >> 16))
                       : "memory");
          if (brow != nullptr) {
            if (!band) {
              acc_lo += ds.x + ds.y;
            } else {
#pragma unroll
              for (int e = 0; e < 2; ++e) {
                const int rel = q + e - j;
                const float v = e ? ds.y : ds.x;
                if (rel <= -R) acc_lo += v;
                else if (rel >= R) acc_hi += v;
                else if (v != 0.f) atomicAdd(part + rel + R, dbias_fixed(v));
              }
            }
          }
        }
        // P^T over S^T and dS^T over dP^T: columns [c0 / 2, c0 / 2 + 8) were read above
        tmem_st8(t_s + c0 / 2, ppk);
        tmem_st8(t_dp + c0 / 2, dpk);
      }
      tmem_st_wait();
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive_warp(&bars->pds_full[db]);
    }
    if (!ok) break;
    if (part != nullptr) {
      // the clamped mass of this unit: one fixed-point red per warp and table end
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
}

// ---------------------------------------------------------- epilogue warps
template <int D, int NQ>
__device__ void bsq_epilogue(const BwdParams& p, uint8_t* smem, BsqBars* bars, uint32_t tmem, int n_units,
                             Fail fail) {
  using C = BsqCfg<D, NQ>;
  const int quad = (threadIdx.x >> 5) & 3;
  const int lr = threadIdx.x & 31;
  const int r = quad * 32 + lr;  // TMEM lane: key row (dV, dK) or column of d (dQ^T)
  const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
  const int H = p.heads;
  uint32_t acc_n = 0, dq_n = 0;
  for (int rr = 0;; ++rr) {
    const int idx = unit_index(rr, blockIdx.x, gridDim.x);
    if (idx >= n_units) break;
    const BsqUnit u = bsq_unit(p, idx);
    if (u.nt == 0) continue;
    bool ok = true;
    for (int t = 0; t < u.nt; ++t) {
      if (!(ok = mbar_wait(&bars->acc_full, acc_n & 1, fail))) break;
      ++acc_n;
      tc_fence_after();
      const int rows = min(kTile, u.seg.lkv - (u.t0 + t) * kTile);
      const int64_t row0 = static_cast<int64_t>(u.seg.k0) + (u.t0 + t) * kTile + quad * 32;  // the warp's first row
      if constexpr (D >= 64) {
        // 64 columns of the warp's 32 rows at a time through its own 4 KB of
        // staging, then four whole 128-byte row pieces per store instruction
        const uint32_t blk = smem_u32(smem + C::kStageOff) + quad * 4096;
#pragma unroll
        for (int part = 0; part < 2 * (D / 64); ++part) {
          const int which = part / (D / 64), hb = part % (D / 64);  // 0: dV, 1: dK
          const float mul = which ? p.scale : 1.0f;
          uint32_t o0[32], o1[32];
          const uint32_t t_acc = tmem + lane_off + (which ? C::kColDk : C::kColDv) + 64 * hb;
          tmem_ld32(t_acc, o0);
          tmem_ld32(t_acc + 32, o1);
          tmem_ld_wait2(o0, o1);
          if (part == 2 * (D / 64) - 1) {  // every column of this tile is in registers
            tc_fence_before();
            mbar_arrive_warp(&bars->acc_empty);
          }
#pragma unroll
          for (int c = 0; c < 64; c += 8) {
            const uint32_t(&o)[32] = c < 32 ? o0 : o1;
            const int cc = c & 31;
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
              w[e] = pack_bf16(__uint_as_float(o[cc + 2 * e]) * mul, __uint_as_float(o[cc + 2 * e + 1]) * mul);
            const int jp = c >> 3;  // 16-byte piece of the 128-byte row piece
            st_shared_v4(blk + lr * 128 + ((jp ^ (lr & 7)) << 4), w[0], w[1], w[2], w[3]);
          }
          __syncwarp();
          __nv_bfloat16* base = which ? p.dk : p.dv;
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const int rw = 4 * k + (lr >> 3), jp = lr & 7;
            uint32_t a, b2, c2, d2;
            ld_shared_v4(blk + rw * 128 + ((jp ^ (rw & 7)) << 4), a, b2, c2, d2);
            if (quad * 32 + rw < rows)
              st_global_v4(base + ((row0 + rw) * H + u.h) * D + 64 * hb + 8 * jp, a, b2, c2, d2);
          }
          __syncwarp();
        }
      } else {
        uint32_t ov[32], ok_[32];
        tmem_ld32(tmem + lane_off + C::kColDv, ov);
        tmem_ld32(tmem + lane_off + C::kColDk, ok_);
        tmem_ld_wait2(ov, ok_);
        tc_fence_before();
        mbar_arrive_warp(&bars->acc_empty);
        if (r < rows) {
          __nv_bfloat16* dv = p.dv + ((row0 + lr) * H + u.h) * D;
          __nv_bfloat16* dk = p.dk + ((row0 + lr) * H + u.h) * D;
#pragma unroll
          for (int c = 0; c < D; c += 8) {
            uint32_t w[4], x[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              w[e] = pack_bf16(__uint_as_float(ov[c + 2 * e]), __uint_as_float(ov[c + 2 * e + 1]));
              x[e] = pack_bf16(__uint_as_float(ok_[c + 2 * e]) * p.scale, __uint_as_float(ok_[c + 2 * e + 1]) * p.scale);
            }
            st_global_v4(dv + c, w[0], w[1], w[2], w[3]);
            st_global_v4(dk + c, x[0], x[1], x[2], x[3]);
          }
        }
      }
    }
    if (!ok) break;
    // the unit's dQ contribution: lane r holds column r of d for every query
    // row, scaled by s, into block (item of this chunk, head) [q_rows][D]
    if (!mbar_wait(&bars->dq_full, dq_n & 1, fail)) break;
    ++dq_n;
    tc_fence_after();
    uint32_t dq[NQ];
    if (quad * 32 < D) {
#pragma unroll
      for (int c0 = 0; c0 < NQ; c0 += 16) {
        uint32_t(&v)[16] = *reinterpret_cast<uint32_t(*)[16]>(dq + c0);
        tmem_ld16(tmem + lane_off + C::kColDq + c0, v);
        tmem_ld_wait16(v);
      }
    }
    tc_fence_before();
    mbar_arrive_warp(&bars->dq_empty);
    if (r < D) {
      const int64_t block = (static_cast<int64_t>(__ldg(p.kv_item_base + u.b)) + u.chunk) * H + u.h;
      float* dst = p.dq_fused + block * p.q_rows * D + r;
#pragma unroll
      for (int q = 0; q < NQ; ++q)
        if (q < p.q_rows) dst[static_cast<int64_t>(q) * D] = __uint_as_float(dq[q]) * p.scale;
    }
  }
}

// ----------------------------------------------------------------- kernel
template <int D, int ACT, int NQ, bool WIN>
__global__ void __launch_bounds__(384, 1) gdpa_bwd_shortq_kernel(const __grid_constant__ BwdParams p) {
  using C = BsqCfg<D, NQ>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  BsqBars* bars = reinterpret_cast<BsqBars*>(smem + C::kBarOff);
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    mbar_init(&bars->qd_full, 1);
    mbar_init(&bars->qd_empty, 1);
    for (int s = 0; s < 4; ++s) {
      mbar_init(&bars->kv_full[s], 1);
      mbar_init(&bars->kv_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars->s_full[s], 1);
      mbar_init(&bars->pds_full[s], 4);
      mbar_init(&bars->ds_empty[s], 1);
    }
    mbar_init(&bars->acc_full, 1);
    mbar_init(&bars->acc_empty, 4);
    mbar_init(&bars->dq_full, 1);
    mbar_init(&bars->dq_empty, 4);
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
  if (warp == 0) bsq_producer<D, NQ>(p, smem, bars, n_units, fail);
  else if (warp == 1) bsq_mma<D, NQ>(p, smem, bars, tmem, n_units, fail);
  else if (warp >= 4 && warp < 8) bsq_act<D, ACT, NQ, WIN>(p, smem, bars, tmem, n_units, fail);
  else if (warp >= 8) bsq_epilogue<D, NQ>(p, smem, bars, tmem, n_units, fail);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

// ------------------------------------------------------------------ launch
#ifndef JGDPA_HEAD_DIM
#error "compile bwd_shortq.cu with -DJGDPA_HEAD_DIM=32, 64 or 128"
#endif

template <int D, int ACT, int NQ>
static cudaError_t launch_bsq_t(const BwdParams& p, int grid, cudaStream_t stream) {
  auto kern = p.window > 0 ? gdpa_bwd_shortq_kernel<D, ACT, NQ, true> : gdpa_bwd_shortq_kernel<D, ACT, NQ, false>;
  // at least half the SM's shared memory: one CTA per SM, so that a second
  // CTA never waits in its TMEM allocation for the first to finish
  constexpr int kSmem = BsqCfg<D, NQ>::kSmemBytes > 120 * 1024 ? BsqCfg<D, NQ>::kSmemBytes : 120 * 1024;
  static DeviceFlags attr_set[2] = {};
  cudaError_t e = smem_attr_once(kern, kSmem, attr_set[p.window > 0]);
  if (e != cudaSuccess) return e;
  kern<<<grid, 384, kSmem, stream>>>(p);
  return cudaGetLastError();
}

// act: 0 GELU, 1 SiLU; nq: the shared query rows, 1..64 (p.q_rows).
template <int D>
cudaError_t launch_bwd_shortq_d(const BwdParams& p, int act, int nq, int grid, cudaStream_t stream) {
  if (nq <= 16) return act == 0 ? launch_bsq_t<D, 0, 16>(p, grid, stream) : launch_bsq_t<D, 1, 16>(p, grid, stream);
  if (nq <= 32) return act == 0 ? launch_bsq_t<D, 0, 32>(p, grid, stream) : launch_bsq_t<D, 1, 32>(p, grid, stream);
  return act == 0 ? launch_bsq_t<D, 0, 64>(p, grid, stream) : launch_bsq_t<D, 1, 64>(p, grid, stream);
}
template cudaError_t launch_bwd_shortq_d<JGDPA_HEAD_DIM>(const BwdParams&, int, int, int, cudaStream_t);

}  // namespace jg
