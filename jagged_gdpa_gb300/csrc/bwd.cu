// Backward jagged GDPA kernels for sm_103a.
//
// The backward is split in two persistent passes so that every output tile
// has exactly one writer and no atomics touch dQ, dK or dV (the split-dQ,
// atomics-free backward of "Eliminating Compute Waste in Asymmetric
// Workloads", aiuniverse.news):
//
//   dkdv pass, unit = (segment, head, 128-row key/value tile j0):
//     for every query tile that meets it:
//       S^T = K Q^T, dP^T = V dO^T                       (tcgen05, TMEM)
//       P^T = act(x)^T, dS^T = dP^T act'(x)^T            (activation warps)
//       (softmax: P = exp(x - LSE_i), dS = P (dP - D_i))
//       dV += P^T dO, dK += dS^T Q                       (tcgen05, TMEM)
//     dK *= s; store dK, dV; dbias partial sums of dS
//   dq pass, unit = (segment, head, 128-row query tile):
//     for every key/value tile: S = Q K^T, dP = dO V^T, dS, dQ += dS K
//     dQ *= s; store
//
// TMEM (512 columns): dkdv uses S^T [0,128), dP^T [128,256), dV [256,256+D),
// dK [256+D, 256+2D); dq uses S [0,128), dP [128,256), dQ [256,256+D).  Two
// activation warpgroups split the 128 columns of a tile; each writes its
// bf16 P / dS over S / dP columns that it has already read, and the MMA picks
// the operand columns per 16-wide K step.
#include "act.cuh"
#include "common.cuh"
#include "ptx.cuh"

namespace jg {

template <int D>
struct BwdCfg {
  static constexpr int kBlockCols = D < 64 ? D : 64;
  static constexpr int kRowBytes = kBlockCols * 2;
  static constexpr int kBlockBytes = kTile * kRowBytes;
  static constexpr int kNumBlocks = D / kBlockCols;
  static constexpr int kTileBytes = kTile * D * 2;
  static constexpr int kStages = D == 128 ? 2 : (D == 64 ? 3 : 4);
  static constexpr uint32_t kSwizzle = kRowBytes == 128 ? 2u : 4u;
  static constexpr int kSBO = 8 * kRowBytes;
  // resident pair (K,V for dkdv / Q,dO for dq), then the streamed pairs
  static constexpr int kResOff = 0;
  static constexpr int kStreamOff = 2 * kTileBytes;
  static constexpr int kBiasOff = kStreamOff + kStages * 2 * kTileBytes;
  static constexpr int kBarOff = kBiasOff + 4 * (kMaxBiasLen + 1);
  static constexpr int kSmemBytes = kBarOff + 512 + 1024;
};

struct BwdBars {
  uint64_t res_full, res_empty;
  uint64_t s_full, p_full, acc_full, acc_empty;
  uint64_t drain;
  uint64_t grp[2];
  uint64_t st_full[4], st_empty[4];
  uint32_t tmem_base;
  int abort;
};

// K-major operand at column offset kk*16 inside a [128][D] tile.
template <int D>
__device__ __forceinline__ uint64_t kmajor_desc(uint32_t tile, int kk) {
  using C = BwdCfg<D>;
  const uint32_t off = (kk * 16 / C::kBlockCols) * C::kBlockBytes + (kk * 16 % C::kBlockCols) * 2;
  return sdesc(tile + off, 16, C::kSBO, C::kSwizzle);
}
// MN-major operand (N = D columns, K = 128 rows) at row offset kk*16.
template <int D>
__device__ __forceinline__ uint64_t mnmajor_desc(uint32_t tile, int kk) {
  using C = BwdCfg<D>;
  return sdesc(tile + kk * 16 * C::kRowBytes, C::kBlockBytes, C::kSBO, C::kSwizzle);
}

// C(tmem) = A_tile(128 x D) * B_tile(128 x D)^T : both K-major.
template <int D>
__device__ __forceinline__ void mma_tile_nt(uint32_t d_tmem, uint32_t a_tile, uint32_t b_tile) {
  constexpr uint32_t idesc = idesc_bf16(kTile, kTile, 0, 0);
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk)
    mma_ss(d_tmem, kmajor_desc<D>(a_tile, kk), kmajor_desc<D>(b_tile, kk), idesc, kk > 0 ? 1u : 0u);
}
// C(tmem, 128 x D) (+)= A(tmem, 128 x 128 bf16, split halves) * B_tile(128 x D, MN-major)
template <int D>
__device__ __forceinline__ void mma_tile_tn(uint32_t d_tmem, uint32_t a_lo, uint32_t a_hi, uint32_t b_tile,
                                            bool accumulate) {
  constexpr uint32_t idesc = idesc_bf16(kTile, D, 0, 1);
#pragma unroll
  for (int kk = 0; kk < kTile / 16; ++kk) {
    const uint32_t a = kk < 4 ? a_lo + kk * 8 : a_hi + (kk - 4) * 8;
    mma_ts(d_tmem, a, mnmajor_desc<D>(b_tile, kk), idesc, (accumulate || kk > 0) ? 1u : 0u);
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

template <bool KV_MAJOR>
__device__ __forceinline__ BwdUnit bwd_unit(const BwdParams& p, int idx) {
  BwdUnit u;
  const Unit w = p.units[idx];
  u.b = w.x;
  u.h = w.y;
  u.tile = w.z;
  u.seg = load_seg(p.q_off, p.kv_off, u.b);
  if constexpr (KV_MAJOR) {
    u.rows = u.seg.lkv - u.tile * kTile;
    u.first = first_q_tile_for_kv_tile(u.tile, p.causal);
    u.count = q_tiles_for_kv_tile(u.tile, u.seg.lq, p.causal);
  } else {
    u.rows = u.seg.lq - u.tile * kTile;
    u.first = 0;
    u.count = kv_tiles_for_q_tile(u.tile, u.seg.lkv, p.causal);
  }
  return u;
}

// ----------------------------------------------------------------- producer
// Resident pair: (K, V) of the unit (dkdv) or (Q, dO) (dq).  Streamed pairs:
// (Q, dO) of each query tile (dkdv) or (K, V) of each key tile (dq).
template <int D, bool KV_MAJOR>
__device__ void bwd_producer(const BwdParams& p, uint8_t* smem, BwdBars* bars, int n_units, Fail fail) {
  using C = BwdCfg<D>;
  const CUtensorMap* res0 = KV_MAJOR ? &p.tm_k : &p.tm_q;
  const CUtensorMap* res1 = KV_MAJOR ? &p.tm_v : &p.tm_do;
  const CUtensorMap* str0 = KV_MAJOR ? &p.tm_q : &p.tm_k;
  const CUtensorMap* str1 = KV_MAJOR ? &p.tm_do : &p.tm_v;
  uint32_t res_it = 0, st_it = 0;
  bool ok = true;
  for (int r = 0; ok; ++r) {
    const int idx = unit_index(r, blockIdx.x, gridDim.x);
    if (idx >= n_units) break;
    const BwdUnit u = bwd_unit<KV_MAJOR>(p, idx);
    if (u.count == 0) continue;
    if (!(ok = mbar_wait(&bars->res_empty, (res_it & 1) ^ 1, fail))) break;
    ++res_it;
    {
      const int row = (KV_MAJOR ? u.seg.k0 : u.seg.q0) + u.tile * kTile;
      mbar_arrive_tx(&bars->res_full, 2 * C::kTileBytes);
      uint8_t* d0 = smem + C::kResOff;
#pragma unroll
      for (int cb = 0; cb < C::kNumBlocks; ++cb) {
        tma_load_3d(d0 + cb * C::kBlockBytes, res0, &bars->res_full, cb * C::kBlockCols, u.h, row);
        tma_load_3d(d0 + C::kTileBytes + cb * C::kBlockBytes, res1, &bars->res_full, cb * C::kBlockCols, u.h,
                    row);
      }
    }
    for (int i = 0; i < u.count; ++i) {
      const int st = st_it % C::kStages;
      if (!(ok = mbar_wait(&bars->st_empty[st], ((st_it / C::kStages) & 1) ^ 1, fail))) break;
      const int row = (KV_MAJOR ? u.seg.q0 : u.seg.k0) + (u.first + i) * kTile;
      mbar_arrive_tx(&bars->st_full[st], 2 * C::kTileBytes);
      uint8_t* d0 = smem + C::kStreamOff + st * 2 * C::kTileBytes;
#pragma unroll
      for (int cb = 0; cb < C::kNumBlocks; ++cb) {
        tma_load_3d(d0 + cb * C::kBlockBytes, str0, &bars->st_full[st], cb * C::kBlockCols, u.h, row);
        tma_load_3d(d0 + C::kTileBytes + cb * C::kBlockBytes, str1, &bars->st_full[st], cb * C::kBlockCols, u.h,
                    row);
      }
      ++st_it;
    }
  }
  if (!ok) {
    if (res_it) mbar_wait_drain(&bars->res_full, (res_it - 1) & 1);
    for (uint32_t i = st_it > C::kStages ? st_it - C::kStages : 0; i < st_it; ++i)
      mbar_wait_drain(&bars->st_full[i % C::kStages], (i / C::kStages) & 1);
  }
}

// ---------------------------------------------------------------- MMA issuer
template <int D, bool KV_MAJOR>
__device__ void bwd_mma(const BwdParams& p, uint8_t* smem, BwdBars* bars, uint32_t tmem, int n_units, Fail fail) {
  using C = BwdCfg<D>;
  const uint32_t res0 = smem_u32(smem + C::kResOff);
  const uint32_t res1 = res0 + C::kTileBytes;
  const uint32_t str_base = smem_u32(smem + C::kStreamOff);
  uint32_t res_it = 0, st_it = 0, p_it = 0, acc_it = 0;
  bool ok = true;
  for (int r = 0; ok; ++r) {
    const int idx = unit_index(r, blockIdx.x, gridDim.x);
    if (idx >= n_units) break;
    const BwdUnit u = bwd_unit<KV_MAJOR>(p, idx);
    if (u.count == 0) continue;
    if (!(ok = mbar_wait(&bars->res_full, res_it & 1, fail))) break;
    ++res_it;
    for (int i = 0; i < u.count; ++i) {
      const int st = st_it % C::kStages;
      const uint32_t s0 = str_base + st * 2 * C::kTileBytes;
      const uint32_t s1 = s0 + C::kTileBytes;
      if (!(ok = mbar_wait(&bars->st_full[st], (st_it / C::kStages) & 1, fail))) break;
      tc_fence_after();
      if constexpr (KV_MAJOR) {
        mma_tile_nt<D>(tmem, res0, s0);        // S^T  = K  Q^T
        mma_tile_nt<D>(tmem + 128, res1, s1);  // dP^T = V  dO^T
      } else {
        mma_tile_nt<D>(tmem, res0, s0);        // S  = Q  K^T
        mma_tile_nt<D>(tmem + 128, res1, s1);  // dP = dO V^T
      }
      mma_commit(&bars->s_full);
      if (i == 0) {
        if (!(ok = mbar_wait(&bars->acc_empty, (acc_it & 1) ^ 1, fail))) break;
        ++acc_it;
      }
      if (!(ok = mbar_wait(&bars->p_full, p_it & 1, fail))) break;
      ++p_it;
      tc_fence_after();
      if constexpr (KV_MAJOR) {
        mma_tile_tn<D>(tmem + 256, tmem + 0, tmem + 64, s1, i > 0);          // dV += P^T  dO
        mma_tile_tn<D>(tmem + 256 + D, tmem + 128, tmem + 192, s0, i > 0);   // dK += dS^T Q
      } else {
        mma_tile_tn<D>(tmem + 256, tmem + 0, tmem + 64, s0, i > 0);          // dQ += dS K
      }
      mma_commit(&bars->st_empty[st]);
      ++st_it;
      if (i == u.count - 1) {
        mma_commit(&bars->acc_full);
        mma_commit(&bars->res_empty);
      }
    }
  }
  mma_commit(&bars->drain);
  mbar_wait_drain(&bars->drain, 0);
}

// --------------------------------------------------------- activation warps
// Element of the bias table for relative position rel.
__device__ __forceinline__ float bias_val(const float* row, int rel, int R) {
  return ld_nc_f32(row + min(max(rel, -R), R) + R);
}

template <int D, int ACT, bool KV_MAJOR>
__device__ void bwd_act(const BwdParams& p, uint8_t* smem, BwdBars* bars, uint32_t tmem, int n_units, Fail fail) {
  using C = BwdCfg<D>;
  constexpr bool kSoftmax = ACT == 2;
  const int warp = threadIdx.x >> 5;
  const int quad = warp & 3;
  const int half = (warp - 4) >> 2;                // which 64 columns this warpgroup owns
  const int r = quad * 32 + (threadIdx.x & 31);    // row of this unit's own tile
  const int act_tid = threadIdx.x - 128;           // 0..255 over both warpgroups
  const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
  const uint32_t t_s = tmem + lane_off + 64 * half;
  const uint32_t t_dp = tmem + lane_off + 128 + 64 * half;
  const int H = p.heads;
  const bool want_dbias = KV_MAJOR && p.dbias_part != nullptr;
  const int R = (p.bias_len - 1) / 2;
  float* sbias = reinterpret_cast<float*>(smem + C::kBiasOff);
  uint32_t s_it = 0, acc_it = 0, grp_it = 0;

  for (int rr = 0;; ++rr) {
    const int idx = unit_index(rr, blockIdx.x, gridDim.x);
    if (idx >= n_units) break;
    const BwdUnit u = bwd_unit<KV_MAJOR>(p, idx);
    if (u.rows <= 0) continue;
    const bool row_ok = r < u.rows;
    const int64_t grow = static_cast<int64_t>(KV_MAJOR ? u.seg.k0 : u.seg.q0) + u.tile * kTile + r;
    const float* brow = p.bias_len ? p.bias + static_cast<int64_t>(u.h) * p.bias_len : nullptr;
    float acc_lo = 0.f, acc_hi = 0.f;  // dbias mass clamped to the table's ends

    if (u.count == 0) {  // no partner rows: the gradient rows are zero
      if (row_ok) {
        if constexpr (KV_MAJOR) {
          __nv_bfloat16* dst = (half == 0 ? p.dv : p.dk) + (grow * H + u.h) * D;
#pragma unroll
          for (int c = 0; c < D; c += 8) st_global_v4(dst + c, 0u, 0u, 0u, 0u);
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
      if (!(ok = mbar_wait(&bars->s_full, s_it & 1, fail))) break;
      ++s_it;
      tc_fence_after();
      const int pt = u.first + i;  // partner tile
      // Geometry: own row index a = tile*128 + r, partner column b = pt*128 + c.
      // rel = i_q - j_kv; valid pairs need j_kv <= i_q under causal masking.
      int lo = 0, hi = kTile;
      int rel0;  // rel at c = 0
      if constexpr (KV_MAJOR) {
        hi = min(kTile, u.seg.lq - pt * kTile);
        if (p.causal && pt == u.tile) lo = r;                 // i >= j  <=>  c >= r
        rel0 = (pt - u.tile) * kTile - r;                      // rel = rel0 + c
      } else {
        hi = min(kTile, u.seg.lkv - pt * kTile);
        if (p.causal && pt == u.tile) hi = min(hi, r + 1);    // j <= i  <=>  c <= r
        rel0 = (u.tile - pt) * kTile + r;                      // rel = rel0 - c
      }
      if (!row_ok) hi = 0;
      const bool tile_masked = lo > 0 || hi < kTile;
      const bool tile_masked_any = __any_sync(0xffffffffu, tile_masked);
      // bias band: is any |rel| < R in this tile?
      const int relmin = (KV_MAJOR ? (pt - u.tile) * kTile - (kTile - 1) : (u.tile - pt) * kTile - (kTile - 1));
      const int relmax = relmin + 2 * (kTile - 1);
      const bool has_bias = brow != nullptr;
      const bool band = has_bias && relmin < R && relmax > -R;
      const float bconst = has_bias ? (relmin >= R ? __ldg(brow + 2 * R) : __ldg(brow)) : 0.f;

#pragma unroll 1
      for (int chunk = 0; chunk < 2; ++chunk) {
        const int cbase = 64 * half + 32 * chunk;  // first column (0..127) of this chunk
        uint32_t sv[32], dpv[32];
        tmem_ld32(t_s + 32 * chunk, sv);
        tmem_ld32(t_dp + 32 * chunk, dpv);
        tmem_ld_wait2(sv, dpv);
        float lse_c[32], del_c[32];
        if constexpr (kSoftmax && KV_MAJOR) {
          // statistics of the query rows that are this chunk's columns
          const int64_t q0 = static_cast<int64_t>(u.h) * p.total_q + u.seg.q0 + pt * kTile + cbase;
          const int lim = max(0, min(32, u.seg.lq - pt * kTile - cbase));
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            lse_c[e] = e < lim ? __ldg(p.lse + q0 + e) * kLog2e : 0.f;
            del_c[e] = e < lim ? __ldg(p.delta + q0 + e) : 0.f;
          }
        }
        uint32_t pk_p[16], pk_ds[16];
        float row_sum = 0.f;
#pragma unroll
        for (int e2 = 0; e2 < 16; ++e2) {
          float pv[2], dsv[2];
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int cl = 2 * e2 + e;
            const int c = cbase + cl;
            const int rel = KV_MAJOR ? rel0 + c : rel0 - c;
            float bias = 0.f;
            if (has_bias) bias = band ? bias_val(brow, rel, R) : bconst;
            const float sval = __uint_as_float(sv[cl]);
            float dp = __uint_as_float(dpv[cl]);
            float pval, ds;
            if constexpr (kSoftmax) {
              const float x2 = __fmaf_rn(sval, p.scale * kLog2e, bias * kLog2e);
              const float lse2 = KV_MAJOR ? lse_c[cl] : lse2_row;
              const float dl = KV_MAJOR ? del_c[cl] : delta_row;
              pval = ex2_sfu(x2 - lse2);
              ds = pval * (dp - dl);
            } else {
              const float x = __fmaf_rn(sval, p.scale, bias);
              float da;
              pval = (chunk == 1 && e2 >= 8) ? act_val_d<ACT, true>(x, da) : act_val_d<ACT, false>(x, da);
              ds = dp * da;
            }
            if (tile_masked_any && (c < lo || c >= hi)) {
              pval = 0.f;
              ds = 0.f;
            }
            pv[e] = pval;
            dsv[e] = ds;
            if (want_dbias) {
              if (band) {
                if (rel >= R) acc_hi += ds;
                else if (rel <= -R) acc_lo += ds;
                else atomicAdd(sbias + rel + R, ds);
              } else {
                row_sum += ds;
              }
            }
          }
          pk_p[e2] = pack_bf16(pv[0], pv[1]);
          pk_ds[e2] = pack_bf16(dsv[0], dsv[1]);
        }
        if (want_dbias && !band) {
          if (relmin >= R) acc_hi += row_sum;
          else acc_lo += row_sum;
        }
        if constexpr (KV_MAJOR) {
          tmem_st16(t_s + 16 * chunk, pk_p);     // P^T over S^T columns already read
          tmem_st16(t_dp + 16 * chunk, pk_ds);   // dS^T over dP^T columns already read
        } else {
          tmem_st16(t_s + 16 * chunk, pk_ds);    // dS over S columns already read
        }
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&bars->p_full);
    }
    if (!ok) break;

    // epilogue
    if (!mbar_wait(&bars->acc_full, acc_it & 1, fail)) break;
    ++acc_it;
    tc_fence_after();
    if constexpr (KV_MAJOR) {
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
      // warpgroup h stores dQ columns [h D/2, (h+1) D/2), scaled by s
      const uint32_t t_acc = tmem + lane_off + 256 + (D / 2) * half;
      __nv_bfloat16* dst = p.dq + (grow * H + u.h) * D + (D / 2) * half;
#pragma unroll
      for (int c0 = 0; c0 < D / 2; c0 += 16) {
        uint32_t o[16];
        tmem_ld16(t_acc + c0, o);
        tmem_ld_wait16(o);
        if (row_ok) {
#pragma unroll
          for (int c = 0; c < 16; c += 8) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
              w[e] = pack_bf16(__uint_as_float(o[c + 2 * e]) * p.scale, __uint_as_float(o[c + 2 * e + 1]) * p.scale);
            st_global_v4(dst + c0 + c, w[0], w[1], w[2], w[3]);
          }
        }
      }
    }
    tc_fence_before();
    mbar_arrive(&bars->acc_empty);

    if (want_dbias) {
      // fold the clamped mass, then flush this unit's partial sums to the
      // CTA's private slice and clear them (bounded group syncs of the 256
      // activation threads)
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        acc_lo += __shfl_xor_sync(0xffffffffu, acc_lo, o);
        acc_hi += __shfl_xor_sync(0xffffffffu, acc_hi, o);
      }
      if ((threadIdx.x & 31) == 0) {
        atomicAdd(sbias, acc_lo);
        atomicAdd(sbias + 2 * R, acc_hi);
      }
      mbar_arrive(&bars->grp[0]);
      if (!mbar_wait(&bars->grp[0], grp_it & 1, fail)) break;
      float* part = p.dbias_part + (static_cast<int64_t>(blockIdx.x) * H + u.h) * p.bias_len;
      for (int e = act_tid; e < p.bias_len; e += 256) {
        part[e] += sbias[e];
        sbias[e] = 0.f;
      }
      mbar_arrive(&bars->grp[1]);
      if (!mbar_wait(&bars->grp[1], grp_it & 1, fail)) break;
      ++grp_it;
    }
  }
}

// ------------------------------------------------------------------- kernel
template <int D, int ACT, bool KV_MAJOR>
__global__ void __launch_bounds__(384, 1) gdpa_bwd_kernel(const __grid_constant__ BwdParams p) {
  using C = BwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  BwdBars* bars = reinterpret_cast<BwdBars*>(smem + C::kBarOff);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(&bars->res_full, 1);
    mbar_init(&bars->res_empty, 1);
    mbar_init(&bars->s_full, 1);
    mbar_init(&bars->p_full, 256);
    mbar_init(&bars->acc_full, 1);
    mbar_init(&bars->acc_empty, 256);
    mbar_init(&bars->drain, 1);
    mbar_init(&bars->grp[0], 256);
    mbar_init(&bars->grp[1], 256);
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&bars->st_full[s], 1);
      mbar_init(&bars->st_empty[s], 1);
    }
    bars->abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&bars->tmem_base, 512);
    tmem_relinquish();
  }
  if (KV_MAJOR && p.dbias_part != nullptr) {  // per-CTA dbias accumulator starts at zero
    float* sbias = reinterpret_cast<float*>(smem + C::kBiasOff);
    for (int e = threadIdx.x; e < p.bias_len; e += blockDim.x) sbias[e] = 0.f;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  int n_units = *p.n_units;
  if (*reinterpret_cast<volatile int*>(p.status) != kOk) n_units = 0;
  Fail fail{&bars->abort, p.status};
  if (warp == 0) {
    if (lane == 0) bwd_producer<D, KV_MAJOR>(p, smem, bars, n_units, fail);
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) bwd_mma<D, KV_MAJOR>(p, smem, bars, tmem, n_units, fail);
    __syncwarp();
  } else if (warp >= 4) {
    bwd_act<D, ACT, KV_MAJOR>(p, smem, bars, tmem, n_units, fail);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

// delta_i = <dO_i, O_i> per (row, head), fp32 from bf16 (softmax backward).
template <int D>
__global__ void softmax_delta_kernel(const __nv_bfloat16* __restrict__ out, const __nv_bfloat16* __restrict__ dout,
                                     float* __restrict__ delta, int64_t total_q, int heads, const int* status) {
  const int64_t row = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;  // row * heads + h
  if (row >= total_q * heads || *status != kOk) return;
  const uint4* o4 = reinterpret_cast<const uint4*>(out + row * D);
  const uint4* d4 = reinterpret_cast<const uint4*>(dout + row * D);
  float acc = 0.f;
#pragma unroll 4
  for (int c = 0; c < D / 8; ++c) {
    const uint4 a = __ldg(o4 + c), b = __ldg(d4 + c);
    const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, bw[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      acc = __fmaf_rn(__uint_as_float(aw[e] << 16), __uint_as_float(bw[e] << 16), acc);
      acc = __fmaf_rn(__uint_as_float(aw[e] & 0xFFFF0000u), __uint_as_float(bw[e] & 0xFFFF0000u), acc);
    }
  }
  const int64_t t = row / heads, h = row % heads;
  delta[h * total_q + t] = acc;
}

// dbias[h][e] = sum over CTAs of the per-CTA partial sums, in CTA order.
__global__ void dbias_reduce_kernel(const float* __restrict__ part, float* __restrict__ dbias, int n_parts, int n) {
  const int e = blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= n) return;
  float acc = 0.f;
  for (int c = 0; c < n_parts; ++c) acc += part[static_cast<int64_t>(c) * n + e];
  dbias[e] = acc;
}

// ------------------------------------------------------------------- launch
template <int D, int ACT, bool KV_MAJOR>
static cudaError_t launch_bwd_t(const BwdParams& p, int grid, cudaStream_t stream) {
  using C = BwdCfg<D>;
  auto kern = gdpa_bwd_kernel<D, ACT, KV_MAJOR>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  kern<<<grid, 384, C::kSmemBytes, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_bwd_pass(const BwdParams& p, int head_dim, int act, bool kv_major, int grid,
                            cudaStream_t stream) {
#define JG_BWD_CASE(DD)                                                                         \
  if (head_dim == DD) {                                                                         \
    if (kv_major) {                                                                             \
      if (act == 0) return launch_bwd_t<DD, 0, true>(p, grid, stream);                          \
      if (act == 1) return launch_bwd_t<DD, 1, true>(p, grid, stream);                          \
      return launch_bwd_t<DD, 2, true>(p, grid, stream);                                        \
    }                                                                                           \
    if (act == 0) return launch_bwd_t<DD, 0, false>(p, grid, stream);                           \
    if (act == 1) return launch_bwd_t<DD, 1, false>(p, grid, stream);                           \
    return launch_bwd_t<DD, 2, false>(p, grid, stream);                                         \
  }
  JG_BWD_CASE(128)
  JG_BWD_CASE(64)
  JG_BWD_CASE(32)
#undef JG_BWD_CASE
  return cudaErrorInvalidValue;
}

cudaError_t launch_softmax_delta(const void* out, const void* dout, float* delta, int64_t total_q, int heads,
                                 int head_dim, const int* status, cudaStream_t stream) {
  const int64_t rows = total_q * heads;
  if (rows == 0) return cudaSuccess;
  const int threads = 256;
  const unsigned blocks = static_cast<unsigned>((rows + threads - 1) / threads);
  const auto* o = static_cast<const __nv_bfloat16*>(out);
  const auto* d = static_cast<const __nv_bfloat16*>(dout);
  if (head_dim == 128) softmax_delta_kernel<128><<<blocks, threads, 0, stream>>>(o, d, delta, total_q, heads, status);
  else if (head_dim == 64) softmax_delta_kernel<64><<<blocks, threads, 0, stream>>>(o, d, delta, total_q, heads, status);
  else softmax_delta_kernel<32><<<blocks, threads, 0, stream>>>(o, d, delta, total_q, heads, status);
  return cudaGetLastError();
}

cudaError_t launch_dbias_reduce(const float* part, float* dbias, int n_parts, int n, cudaStream_t stream) {
  if (n == 0) return cudaSuccess;
  dbias_reduce_kernel<<<(n + 255) / 256, 256, 0, stream>>>(part, dbias, n_parts, n);
  return cudaGetLastError();
}

}  // namespace jg
