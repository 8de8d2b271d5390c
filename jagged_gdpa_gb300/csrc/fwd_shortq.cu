// Short-query forward for sm_103a: every segment has at most NQ <= 64 query
// rows (PMA-style pooling, where a few learned seed queries are shared by
// every segment: "GEM Training: How Meta Doubled the Efficiency of Its ..."
// (globalainews.in), section "What to watch").
//
// With 128 query rows per MMA, a segment of 16 queries would leave 7/8 of
// every S tile and of its activation dead.  Here the keys take the MMA's 128
// rows instead (swap-AB): S^T = K Q^T is 128 keys x NQ queries, so the
// activation touches only live elements.  Each activation thread owns one key
// row of the tile and writes its NQ values of P, transposed, into a shared
// P tile [128 query rows][128 keys] (rows >= NQ never written and their O
// rows never stored), which is the A operand of O += P V (M = 128).
//
// A persistent CTA walks (segment, head) units longest first; a unit streams
// every key/value tile of its segment once.  Warp roles:
//   warp 0      TMA producer: the unit's query block, K/V tiles into a ring
//   warp 1      MMA issuer: S^T = K Q^T (N = NQ) into one of two TMEM
//               buffers, O += P V from the shared P tiles; owns TMEM
//   warps 4-7   activation (one key row per thread) and the O epilogue
// TMEM: S^T buffers [0, NQ) and [NQ, 2 NQ), O [128, 128 + D).
//
// GELU / SiLU only (no normalisation, so no running row statistics); the
// launcher sends softmax to the general forward kernel.
#include "act.cuh"
#include "common.cuh"
#include "ptx.cuh"

namespace jg {

template <int D>
struct SqCfg {
  static constexpr int kBlockCols = D < 64 ? D : 64;
  static constexpr int kRowBytes = kBlockCols * 2;
  static constexpr int kBlockBytes = kTile * kRowBytes;
  static constexpr int kNumBlocks = D / kBlockCols;
  static constexpr int kTileBytes = kTile * D * 2;
  static constexpr int kStages = D == 128 ? 2 : 3;
  static constexpr uint32_t kSwizzle = kRowBytes == 128 ? 2u : 4u;
  static constexpr int kSBO = 8 * kRowBytes;
  static constexpr int kPBytes = kTile * kTile * 2;  // one P tile, two 64-key column blocks
  static constexpr int kPOff = 0;                    // two P tiles (1024-aligned)
  static constexpr int kQOff = kPOff + 2 * kPBytes;
  static constexpr int kKOff = kQOff + kTileBytes;
  static constexpr int kVOff = kKOff + kStages * kTileBytes;
  static constexpr int kBarOff = kVOff + kStages * kTileBytes;
  static constexpr int kSmemBytes = kBarOff + 512 + 1024;
  static_assert(kSmemBytes <= 232448, "shared memory per CTA");
};

struct SqBars {
  uint64_t q_full, q_empty;
  uint64_t k_full[3], k_empty[3], v_full[3], v_empty[3];
  uint64_t s_full[2], s_empty[2], p_full[2], p_empty[2];
  uint64_t o_full, o_empty;
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};

// Key tiles [k0, k0 + nkv) of the unit's single query block (tile 0).
struct SqUnit {
  int b, h;
  Seg seg;
  int k0, nkv;
};

template <bool WIN>
__device__ __forceinline__ SqUnit sq_unit(const FwdParams& p, int idx) {
  SqUnit u;
  const Unit w = p.units[idx];
  u.b = w.x;
  u.h = w.y;
  u.seg = load_seg(p.q_off, p.kv_off, u.b);
  const TileSpan sp = u.seg.lq > 0 ? kv_span_for_q_tile(0, u.seg.lkv, p.causal, WIN ? p.window : 0)
                                   : TileSpan{0, 0};
  u.k0 = sp.first;
  u.nkv = sp.count;
  return u;
}

// ------------------------------------------------------------- producer
template <int D, bool WIN>
__device__ void sq_producer(const FwdParams& p, uint8_t* smem, SqBars* bars, int n_units, Fail fail) {
  using C = SqCfg<D>;
  uint32_t q_it = 0, kv_it = 0, k_it = 0;
  const bool leader = elect_one();
  bool ok = true;
  for (int r = 0; ok; ++r) {
    const int idx = unit_index(r, blockIdx.x, gridDim.x);
    if (idx >= n_units) break;
    const SqUnit u = sq_unit<WIN>(p, idx);
    if (u.nkv == 0) continue;
    if (!(ok = mbar_wait_warp(&bars->q_empty, (q_it & 1) ^ 1, fail))) break;
    if (leader) {
      mbar_arrive_tx(&bars->q_full, C::kTileBytes);
      const int row = p.q_shared ? 0 : u.seg.q0;  // a 128-row box: rows past the block are unused
#pragma unroll
      for (int cb = 0; cb < C::kNumBlocks; ++cb)
        tma_load_3d(smem + C::kQOff + cb * C::kBlockBytes, &p.tm_q, &bars->q_full, cb * C::kBlockCols, u.h, row);
    }
    ++q_it;
    for (int kt = 0; kt < u.nkv && ok; ++kt) {
      const int st = kv_it % C::kStages;
      const uint32_t empty_phase = ((kv_it / C::kStages) & 1) ^ 1;
      const int row = u.seg.k0 + (u.k0 + kt) * kTile;
      if (!(ok = mbar_wait_warp(&bars->k_empty[st], empty_phase, fail))) break;
      if (leader) {
        mbar_arrive_tx(&bars->k_full[st], C::kTileBytes);
#pragma unroll
        for (int cb = 0; cb < C::kNumBlocks; ++cb)
          tma_load_3d(smem + C::kKOff + st * C::kTileBytes + cb * C::kBlockBytes, &p.tm_k, &bars->k_full[st],
                      cb * C::kBlockCols, u.h, row);
      }
      ++k_it;
      if (!(ok = mbar_wait_warp(&bars->v_empty[st], empty_phase, fail))) break;
      if (leader) {
        mbar_arrive_tx(&bars->v_full[st], C::kTileBytes);
#pragma unroll
        for (int cb = 0; cb < C::kNumBlocks; ++cb)
          tma_load_3d(smem + C::kVOff + st * C::kTileBytes + cb * C::kBlockBytes, &p.tm_v, &bars->v_full[st],
                      cb * C::kBlockCols, u.h, row);
      }
      ++kv_it;
    }
  }
  if (!ok) {  // let the copies already issued land before the CTA exits
    if (q_it) mbar_wait_drain(&bars->q_full, (q_it - 1) & 1);
    for (uint32_t i = k_it > C::kStages ? k_it - C::kStages : 0; i < k_it; ++i)
      mbar_wait_drain(&bars->k_full[i % C::kStages], (i / C::kStages) & 1);
    for (uint32_t i = kv_it > C::kStages ? kv_it - C::kStages : 0; i < kv_it; ++i)
      mbar_wait_drain(&bars->v_full[i % C::kStages], (i / C::kStages) & 1);
  }
}

// ------------------------------------------------------------ MMA issuer
// S^T (TMEM, 128 keys x NQ) = K (128 x D, K-major) * Q_block^T (NQ x D, K-major).
template <int D, int NQ>
__device__ __forceinline__ void sq_issue_s(uint32_t d_tmem, uint32_t k_addr, uint32_t q_addr, bool leader) {
  using C = SqCfg<D>;
  constexpr uint32_t idesc = idesc_bf16(kTile, NQ, 0, 0);
  const uint64_t a0 = sdesc(k_addr, 16, C::kSBO, C::kSwizzle), b0 = sdesc(q_addr, 16, C::kSBO, C::kSwizzle);
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint64_t off = static_cast<uint64_t>((kk * 16 / C::kBlockCols) * C::kBlockBytes +
                                               (kk * 16 % C::kBlockCols) * 2) >> 4;
    if (leader) mma_ss(d_tmem, a0 + off, b0 + off, idesc, kk > 0 ? 1u : 0u);
  }
}
// O (TMEM, 128 x D) (+)= P (128 x 128 keys, K-major, 128-byte swizzle) * V (128 keys x D, MN-major).
template <int D>
__device__ __forceinline__ void sq_issue_pv(uint32_t d_tmem, uint32_t p_addr, uint32_t v_addr, bool accumulate,
                                            bool leader) {
  using C = SqCfg<D>;
  constexpr uint32_t idesc = idesc_bf16(kTile, D, 0, 1);
  const uint64_t a0 = sdesc(p_addr, 16, 8 * 128, 2u), b0 = sdesc(v_addr, C::kBlockBytes, C::kSBO, C::kSwizzle);
#pragma unroll
  for (int kk = 0; kk < kTile / 16; ++kk) {
    const uint64_t aoff = static_cast<uint64_t>((kk * 16 / 64) * (kTile * 128) + (kk * 16 % 64) * 2) >> 4;
    const uint64_t boff = static_cast<uint64_t>(kk * 16 * C::kRowBytes) >> 4;
    if (leader) mma_ss(d_tmem, a0 + aoff, b0 + boff, idesc, (accumulate || kk > 0) ? 1u : 0u);
  }
}

template <int D, int NQ, bool WIN>
__device__ void sq_mma(const FwdParams& p, uint8_t* smem, SqBars* bars, uint32_t tmem, int n_units, Fail fail) {
  using C = SqCfg<D>;
  const uint32_t q_addr = smem_u32(smem + C::kQOff);
  const uint32_t k_base = smem_u32(smem + C::kKOff), v_base = smem_u32(smem + C::kVOff);
  const uint32_t p_base = smem_u32(smem + C::kPOff);
  uint32_t q_it = 0, kv_it = 0, s_n = 0, p_n = 0, o_n = 0;
  const bool leader = elect_one();
  bool ok = true;
  for (int r = 0; ok; ++r) {
    const int idx = unit_index(r, blockIdx.x, gridDim.x);
    if (idx >= n_units) break;
    const SqUnit u = sq_unit<WIN>(p, idx);
    if (u.nkv == 0) continue;
    if (!(ok = mbar_wait_warp(&bars->q_full, q_it & 1, fail))) break;
    ++q_it;
    // S^T of key tile t goes to TMEM buffer (s_n % 2) once the activation
    // warps have read that buffer's previous tile
    auto issue_s = [&](uint32_t it) -> bool {
      const int st = it % C::kStages, sb = s_n & 1;
      if (!mbar_wait_warp(&bars->s_empty[sb], ((s_n >> 1) & 1) ^ 1, fail)) return false;
      if (!mbar_wait_warp(&bars->k_full[st], (it / C::kStages) & 1, fail)) return false;
      tc_fence_after();
      sq_issue_s<D, NQ>(tmem + NQ * sb, k_base + st * C::kTileBytes, q_addr, leader);
      if (leader) mma_commit(&bars->s_full[sb]);
      if (leader) mma_commit(&bars->k_empty[st]);
      ++s_n;
      return true;
    };
    if (!(ok = issue_s(kv_it))) break;
    for (int kt = 0; kt < u.nkv && ok; ++kt) {
      const uint32_t it = kv_it + kt;
      if (kt + 1 < u.nkv) {
        if (!(ok = issue_s(it + 1))) break;
      } else if (leader) {
        mma_commit(&bars->q_empty);  // every S^T of the unit issued
      }
      if (kt == 0) {  // the previous unit's O has been read
        if (!(ok = mbar_wait_warp(&bars->o_empty, (o_n & 1) ^ 1, fail))) break;
        ++o_n;
      }
      const int st = it % C::kStages, pb = p_n & 1;
      if (!(ok = mbar_wait_warp(&bars->p_full[pb], (p_n >> 1) & 1, fail))) break;
      if (!(ok = mbar_wait_warp(&bars->v_full[st], (it / C::kStages) & 1, fail))) break;
      tc_fence_after();
      sq_issue_pv<D>(tmem + 128, p_base + pb * C::kPBytes, v_base + st * C::kTileBytes, kt > 0, leader);
      if (leader) mma_commit(&bars->p_empty[pb]);
      if (leader) mma_commit(&bars->v_empty[st]);
      ++p_n;
    }
    if (!ok) break;
    kv_it += u.nkv;
    if (leader) mma_commit(&bars->o_full);
  }
  if (leader) mma_commit(&bars->drain);
  mbar_wait_drain(&bars->drain, 0);
}

// ------------------------------------------------------ activation warps
// Byte offset of element (query row q, key column c) in a P tile: two
// 64-key column blocks of [128 rows][128 bytes], 16-byte pieces swizzled by
// the row (the layout TMA writes and the MMA descriptor reads).
__device__ __forceinline__ uint32_t sq_p_offset(int q, int c) {
  return (c >> 6) * (kTile * 128) + q * 128 + ((((c & 63) >> 3) ^ (q & 7)) << 4) + (c & 7) * 2;
}

template <int D, int ACT, int NQ, bool WIN>
__device__ void sq_act(const FwdParams& p, uint8_t* smem, SqBars* bars, uint32_t tmem, int n_units, Fail fail) {
  using C = SqCfg<D>;
  const int warp = threadIdx.x >> 5;
  const int quad = warp & 3;
  const int r = quad * 32 + (threadIdx.x & 31);  // key row of the tile (S^T lane), query row of O
  const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
  const uint32_t p_base = smem_u32(smem + C::kPOff);
  const int H = p.heads;
  uint32_t s_n = 0, p_n = 0, o_n = 0;
  const float hs = 0.5f * p.scale;
  for (int rr = 0;; ++rr) {
    const int idx = unit_index(rr, blockIdx.x, gridDim.x);
    if (idx >= n_units) break;
    const SqUnit u = sq_unit<WIN>(p, idx);
    if (u.seg.lq <= 0) continue;
    const int64_t q_row0 = u.seg.q0;  // the segment's first output row
    if (u.nkv == 0) {  // no keys: O = 0
      if (r < u.seg.lq) {
        __nv_bfloat16* dst = p.out + ((q_row0 + r) * H + u.h) * D;
#pragma unroll
        for (int c = 0; c < D; c += 8) st_global_v4(dst + c, 0u, 0u, 0u, 0u);
      }
      continue;
    }
    const float* brow = p.bias_len ? p.bias + static_cast<int64_t>(u.h) * p.bias_len : nullptr;
    const int R = (p.bias_len - 1) / 2;
    bool ok = true;
    for (int kt = u.k0; kt < u.k0 + u.nkv; ++kt) {
      const int sb = s_n & 1;
      if (!(ok = mbar_wait(&bars->s_full[sb], (s_n >> 1) & 1, fail))) break;
      tc_fence_after();
      uint32_t sv[NQ];
      if constexpr (NQ == 16) {
        uint32_t(&v)[16] = *reinterpret_cast<uint32_t(*)[16]>(sv);
        tmem_ld16(tmem + lane_off + NQ * sb, v);
        tmem_ld_wait16(v);
      } else {
#pragma unroll
        for (int c0 = 0; c0 < NQ; c0 += 32) {
          uint32_t(&v)[32] = *reinterpret_cast<uint32_t(*)[32]>(sv + c0);
          tmem_ld32(tmem + lane_off + NQ * sb + c0, v);
          tmem_ld_wait(v);
        }
      }
      tc_fence_before();
      mbar_arrive_warp(&bars->s_empty[sb]);
      ++s_n;
      // key j = kt 128 + r against query i (column q): valid when j < Lkv,
      // i < Lq, causal j <= i, window |i - j| < w; bias index clamp(i - j)
      const int j = kt * kTile + r;
      const bool j_ok = j < u.seg.lkv;
      uint16_t pv[NQ];
#pragma unroll
      for (int q = 0; q < NQ; q += 2) {
        float2 bias = f2(0.f);
        if (brow != nullptr)
          bias = make_float2(ld_nc_f32(brow + min(max(q - j, -R), R) + R),
                             ld_nc_f32(brow + min(max(q + 1 - j, -R), R) + R));
        float2 hx = __ffma2_rn(make_float2(__uint_as_float(sv[q]), __uint_as_float(sv[q + 1])), f2(hs),
                               __fmul2_rn(bias, f2(0.5f)));
        bool ok0 = j_ok && q < u.seg.lq, ok1 = j_ok && q + 1 < u.seg.lq;
        if (p.causal) {
          ok0 = ok0 && j <= q;
          ok1 = ok1 && j <= q + 1;
        }
        if constexpr (WIN) {
          ok0 = ok0 && abs(q - j) < p.window;
          ok1 = ok1 && abs(q + 1 - j) < p.window;
        }
        if (!ok0) hx.x = 0.f;  // act(0) = 0
        if (!ok1) hx.y = 0.f;
        const float2 y = act2_route<ACT, 0>(hx);
        const uint32_t pk = pack_bf16(y.x, y.y);
        pv[q] = static_cast<uint16_t>(pk & 0xFFFFu);
        pv[q + 1] = static_cast<uint16_t>(pk >> 16);
      }
      // P[i][j] for the NQ query rows into a free P tile, transposed
      const int pb = p_n & 1;
      if (!(ok = mbar_wait(&bars->p_empty[pb], ((p_n >> 1) & 1) ^ 1, fail))) break;
      const uint32_t pt = p_base + pb * C::kPBytes;
#pragma unroll
      for (int q = 0; q < NQ; ++q)
        asm volatile("st.shared.u16 [%0], %1;" ::"r"(pt + sq_p_offset(q, r)), "h"(pv[q]) : "memory");
      fence_proxy_async_smem();
      mbar_arrive_warp(&bars->p_full[pb]);
      ++p_n;
    }
    if (!ok) break;
    // epilogue: O rows < Lq (TMEM lane = query row) -> bf16 -> global
    if (!mbar_wait(&bars->o_full, o_n & 1, fail)) break;
    ++o_n;
    tc_fence_after();
    __nv_bfloat16* dst = p.out + ((q_row0 + r) * H + u.h) * D;
#pragma unroll
    for (int c0 = 0; c0 < D; c0 += 32) {
      uint32_t o[32];
      tmem_ld32(tmem + lane_off + 128 + c0, o);
      tmem_ld_wait(o);
      if (r < u.seg.lq) {
#pragma unroll
        for (int c = 0; c < 32; c += 8) {
          uint32_t w[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) w[e] = pack_bf16(__uint_as_float(o[c + 2 * e]), __uint_as_float(o[c + 2 * e + 1]));
          st_global_v4(dst + c0 + c, w[0], w[1], w[2], w[3]);
        }
      }
    }
    tc_fence_before();
    mbar_arrive_warp(&bars->o_empty);
  }
}

// ----------------------------------------------------------------- kernel
template <int D, int ACT, int NQ, bool WIN>
__global__ void __launch_bounds__(256, 1) gdpa_fwd_shortq_kernel(const __grid_constant__ FwdParams p) {
  using C = SqCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  SqBars* bars = reinterpret_cast<SqBars*>(smem + C::kBarOff);
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 1);
    mbar_init(&bars->q_empty, 1);
    for (int s = 0; s < 3; ++s) {
      mbar_init(&bars->k_full[s], 1);
      mbar_init(&bars->k_empty[s], 1);
      mbar_init(&bars->v_full[s], 1);
      mbar_init(&bars->v_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars->s_full[s], 1);
      mbar_init(&bars->s_empty[s], 4);
      mbar_init(&bars->p_full[s], 4);
      mbar_init(&bars->p_empty[s], 1);
    }
    mbar_init(&bars->o_full, 1);
    mbar_init(&bars->o_empty, 4);
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
  if (warp == 0) sq_producer<D, WIN>(p, smem, bars, n_units, fail);
  else if (warp == 1) sq_mma<D, NQ, WIN>(p, smem, bars, tmem, n_units, fail);
  else if (warp >= 4) sq_act<D, ACT, NQ, WIN>(p, smem, bars, tmem, n_units, fail);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 256);
}

// ------------------------------------------------------------------ launch
#ifndef JGDPA_HEAD_DIM
#error "compile fwd_shortq.cu with -DJGDPA_HEAD_DIM=32, 64 or 128"
#endif

template <int D, int ACT, int NQ>
static cudaError_t launch_sq_t(const FwdParams& p, int grid, cudaStream_t stream) {
  auto kern = p.window > 0 ? gdpa_fwd_shortq_kernel<D, ACT, NQ, true> : gdpa_fwd_shortq_kernel<D, ACT, NQ, false>;
  constexpr int kSmem = SqCfg<D>::kSmemBytes;
  static DeviceFlags attr_set[2] = {};
  cudaError_t e = smem_attr_once(kern, kSmem, attr_set[p.window > 0]);
  if (e != cudaSuccess) return e;
  kern<<<grid, 256, kSmem, stream>>>(p);
  return cudaGetLastError();
}

// act: 0 GELU, 1 SiLU; nq: the query rows of every segment, 1..64.
template <int D>
cudaError_t launch_fwd_shortq_d(const FwdParams& p, int act, int nq, int grid, cudaStream_t stream) {
  if (nq <= 16) return act == 0 ? launch_sq_t<D, 0, 16>(p, grid, stream) : launch_sq_t<D, 1, 16>(p, grid, stream);
  if (nq <= 32) return act == 0 ? launch_sq_t<D, 0, 32>(p, grid, stream) : launch_sq_t<D, 1, 32>(p, grid, stream);
  return act == 0 ? launch_sq_t<D, 0, 64>(p, grid, stream) : launch_sq_t<D, 1, 64>(p, grid, stream);
}
template cudaError_t launch_fwd_shortq_d<JGDPA_HEAD_DIM>(const FwdParams&, int, int, int, cudaStream_t);

}  // namespace jg
