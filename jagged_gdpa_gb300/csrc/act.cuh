// Device activations of the GDPA kernels: GELU and SiLU with their
// derivatives, by two routes that give the same function up to rounding.
//
//  * SFU route: sigmoid(z) = 1/2 + tanh(z/2)/2 with the hardware tanh
//    (tanh.approx.f32, one special-function-unit op per element).
//  * ALU route: sigmoid(z) = 1/(1 + 2^(-z log2 e)) with 2^w from a polynomial
//    after range reduction and 1/a from an integer seed plus two Newton
//    steps -- FMA/integer pipes only, no special-function unit.
//
// The GDPA kernel redesign replaces the activation's special-function-unit
// work by an ALU-only polynomial to remove SFU contention ("Meta redesigns
// AI training infrastructure ...", aiuniverse.news, section "Custom Kernels
// and 5D Parallelism for Trillion-Parameter Scale": a 6th-order Taylor
// expansion).  The pages give neither the expanded function nor the range
// reduction; here GELU is evaluated as x * sigmoid(a x + b x^3) and the
// kernels send a fixed share of each tile through the ALU route and the rest
// through the SFU route, so that neither pipe is the bottleneck.
//
// Constants come from fit_constants.py (next to this file):
//   a, b      minimise max |x sigmoid(a x + b x^3) - x Phi(x)| on [-16, 16]
//             (2.71e-4; the classic tanh-form constants give 4.73e-4)
//   P0..P3    degree-3 minimax fit of 2^f on [-1/2, 1/2] (rel. err 1.1e-4)
//   kRcpSeed  integer seed for 1/a (rel. err 5.1e-2 before the Newton steps)
#pragma once

#include <cstdint>

namespace jg {

constexpr float kGeluA = 1.60031416f;
constexpr float kGeluB = 0.0694017869f;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kExpP0 = 0.999941753f;
constexpr float kExpP1 = 0.693257044f;
constexpr float kExpP2 = 0.242413568f;
constexpr float kExpP3 = 0.055092146f;
constexpr int kRcpSeed = 0x7EF311C2;

__device__ __forceinline__ float tanh_sfu(float x) {
  float y;
  asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float ex2_sfu(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// 2^w for w in [-64, 64]: w = n + f with integer n and |f| <= 1/2, 2^f from
// the polynomial, 2^n added to the exponent field.
__device__ __forceinline__ float exp2_alu(float w) {
  const float kRound = 12582912.0f;  // 1.5 * 2^23: adding it rounds to an integer
  const float t = __fadd_rn(w, kRound);
  const float n = __fsub_rn(t, kRound);
  const float f = __fsub_rn(w, n);
  float p = __fmaf_rn(kExpP3, f, kExpP2);
  p = __fmaf_rn(p, f, kExpP1);
  p = __fmaf_rn(p, f, kExpP0);
  return __int_as_float(__float_as_int(p) + (__float_as_int(t) << 23));
}

// 1/a for a >= 1 (finite): seed by integer subtraction, then two Newton steps.
__device__ __forceinline__ float rcp_alu(float a) {
  float y = __int_as_float(kRcpSeed - __float_as_int(a));
  float e = __fmaf_rn(-a, y, 1.0f);
  y = __fmaf_rn(y, e, y);
  e = __fmaf_rn(-a, y, 1.0f);
  return __fmaf_rn(y, e, y);
}

// sigmoid(z) and 2^(-z log2 e) by the ALU route; z given as w = -z log2 e.
__device__ __forceinline__ float sigmoid_alu_w(float w, float& e) {
  w = fminf(fmaxf(w, -64.0f), 64.0f);
  e = exp2_alu(w);
  return rcp_alu(1.0f + e);
}

// ----------------------------------------------------------------- GELU
__device__ __forceinline__ float gelu_sfu(float x) {
  const float x2 = x * x;
  const float u = x * __fmaf_rn(0.5f * kGeluB, x2, 0.5f * kGeluA);
  const float t = tanh_sfu(u);
  const float hx = 0.5f * x;
  return __fmaf_rn(hx, t, hx);
}
__device__ __forceinline__ float gelu_sfu_d(float x, float& dy) {
  const float x2 = x * x;
  const float u = x * __fmaf_rn(0.5f * kGeluB, x2, 0.5f * kGeluA);
  const float t = tanh_sfu(u);
  const float hx = 0.5f * x;
  // d/dx [x s(k(x))] = s + x s (1-s) k',  s = (1+t)/2,  s(1-s) = (1-t^2)/4
  const float q = __fmaf_rn(-t, t, 1.0f);
  const float s = __fmaf_rn(0.5f, t, 0.5f);
  const float kp = __fmaf_rn(0.5f * 3.0f * kGeluB, x2, 0.5f * kGeluA);  // k'/2
  dy = __fmaf_rn(hx * q, kp, s);
  return __fmaf_rn(hx, t, hx);
}
__device__ __forceinline__ float gelu_alu(float x) {
  const float x2 = x * x;
  const float w = x * __fmaf_rn(-kGeluB * kLog2e, x2, -kGeluA * kLog2e);
  float e;
  const float s = sigmoid_alu_w(w, e);
  return x * s;
}
__device__ __forceinline__ float gelu_alu_d(float x, float& dy) {
  const float x2 = x * x;
  const float w = x * __fmaf_rn(-kGeluB * kLog2e, x2, -kGeluA * kLog2e);
  float e;
  const float s = sigmoid_alu_w(w, e);
  // s (1 - s) = e s^2
  const float kp = __fmaf_rn(3.0f * kGeluB, x2, kGeluA);
  dy = s * __fmaf_rn(x * e * s, kp, 1.0f);
  return x * s;
}

// ----------------------------------------------------------------- SiLU
__device__ __forceinline__ float silu_sfu(float x) {
  const float hx = 0.5f * x;
  const float t = tanh_sfu(hx);
  return __fmaf_rn(hx, t, hx);
}
__device__ __forceinline__ float silu_sfu_d(float x, float& dy) {
  const float hx = 0.5f * x;
  const float t = tanh_sfu(hx);
  // s + x s (1-s) = (1+t)/2 + x (1-t^2)/4
  const float q = __fmaf_rn(-t, t, 1.0f);
  const float s = __fmaf_rn(0.5f, t, 0.5f);
  dy = __fmaf_rn(0.25f * x, q, s);
  return __fmaf_rn(hx, t, hx);
}
__device__ __forceinline__ float silu_alu(float x) {
  float e;
  const float s = sigmoid_alu_w(-kLog2e * x, e);
  return x * s;
}
__device__ __forceinline__ float silu_alu_d(float x, float& dy) {
  float e;
  const float s = sigmoid_alu_w(-kLog2e * x, e);
  dy = s * __fmaf_rn(x * e, s, 1.0f);
  return x * s;
}

// ------------------------------------------------- packed (two-lane) forms
// Both take hx = x / 2 for two elements (the kernels fold the 1/2 into the
// scale and bias), so GELU(x) = hx + hx tanh(u) with
// u = (a x + b x^3) / 2 = hx (a + 4 b hx^2), and SiLU(x) = hx + hx tanh(hx).
__device__ __forceinline__ float2 f2(float v) { return make_float2(v, v); }

__device__ __forceinline__ float2 tanh2_sfu(float2 u) { return make_float2(tanh_sfu(u.x), tanh_sfu(u.y)); }

// 2^w for two lanes, w already in [-64, 64].
__device__ __forceinline__ float2 exp2_alu2(float2 w) {
  const float kRound = 12582912.0f;
  const float2 t = __fadd2_rn(w, f2(kRound));
  const float2 n = __fadd2_rn(t, f2(-kRound));
  const float2 f = __fadd2_rn(w, make_float2(-n.x, -n.y));
  float2 p = __ffma2_rn(f2(kExpP3), f, f2(kExpP2));
  p = __ffma2_rn(p, f, f2(kExpP1));
  p = __ffma2_rn(p, f, f2(kExpP0));
  return make_float2(__int_as_float(__float_as_int(p.x) + (__float_as_int(t.x) << 23)),
                     __int_as_float(__float_as_int(p.y) + (__float_as_int(t.y) << 23)));
}
// 1 / a for two lanes (a >= 1).
__device__ __forceinline__ float2 rcp_alu2(float2 a) {
  float2 y = make_float2(__int_as_float(kRcpSeed - __float_as_int(a.x)),
                         __int_as_float(kRcpSeed - __float_as_int(a.y)));
  const float2 na = make_float2(-a.x, -a.y);
  float2 e = __ffma2_rn(na, y, f2(1.0f));
  y = __ffma2_rn(y, e, y);
  e = __ffma2_rn(na, y, f2(1.0f));
  return __ffma2_rn(y, e, y);
}
// sigmoid(z) with w = -z log2 e given; also returns e = 2^w.
__device__ __forceinline__ float2 sigmoid_alu2_w(float2 w, float2& e) {
  w = make_float2(fminf(fmaxf(w.x, -64.0f), 64.0f), fminf(fmaxf(w.y, -64.0f), 64.0f));
  e = exp2_alu2(w);
  return rcp_alu2(__fadd2_rn(e, f2(1.0f)));
}

template <int ACT>
__device__ __forceinline__ float2 act2_sfu(float2 hx) {
  float2 u = hx;
  if constexpr (ACT == 0) u = __fmul2_rn(hx, __ffma2_rn(__fmul2_rn(hx, hx), f2(4.0f * kGeluB), f2(kGeluA)));
  return __ffma2_rn(hx, tanh2_sfu(u), hx);
}
template <int ACT>
__device__ __forceinline__ float2 act2_alu(float2 hx) {
  // w = -2 u log2 e  (GELU),  w = -2 hx log2 e  (SiLU);  y = 2 hx sigmoid
  float2 w;
  if constexpr (ACT == 0)
    w = __fmul2_rn(hx, __ffma2_rn(__fmul2_rn(hx, hx), f2(-8.0f * kGeluB * kLog2e), f2(-2.0f * kGeluA * kLog2e)));
  else
    w = __fmul2_rn(hx, f2(-2.0f * kLog2e));
  float2 e;
  const float2 s = sigmoid_alu2_w(w, e);
  const float2 hs = __fmul2_rn(hx, s);
  return __fadd2_rn(hs, hs);
}
template <int ACT, bool ALU>
__device__ __forceinline__ float2 act2(float2 hx) {
  if constexpr (ALU) return act2_alu<ACT>(hx);
  else return act2_sfu<ACT>(hx);
}

// Exponential route: sigmoid(z) = 1 / (1 + 2^(-z log2 e)) with the hardware
// ex2 (twice the special-function rate of tanh on this GPU) and the
// reciprocal from the integer seed plus one Newton step on the FMA pipe
// (relative error 2.6e-3, below the bf16 rounding of P).  Forward only.
__device__ __forceinline__ float2 rcp1_alu2(float2 a) {
  const float2 y = make_float2(__int_as_float(kRcpSeed - __float_as_int(a.x)),
                               __int_as_float(kRcpSeed - __float_as_int(a.y)));
  const float2 e = __ffma2_rn(make_float2(-a.x, -a.y), y, f2(1.0f));
  return __ffma2_rn(y, e, y);
}
template <int ACT>
__device__ __forceinline__ float2 act2_ex2(float2 hx) {
  float2 w;  // w = -k(x) log2 e with x = 2 hx
  if constexpr (ACT == 0)
    w = __fmul2_rn(hx, __ffma2_rn(__fmul2_rn(hx, hx), f2(-8.0f * kGeluB * kLog2e), f2(-2.0f * kGeluA * kLog2e)));
  else
    w = __fmul2_rn(hx, f2(-2.0f * kLog2e));
  // 2^w overflows to +inf for w > 128: then 1 + e = inf and the seed gives a
  // tiny positive y, so sigmoid -> 0 as it should; clamp keeps it finite.
  w = make_float2(fminf(w.x, 64.0f), fminf(w.y, 64.0f));
  const float2 e = make_float2(ex2_sfu(w.x), ex2_sfu(w.y));
  const float2 s = rcp1_alu2(__fadd2_rn(e, f2(1.0f)));
  const float2 hs = __fmul2_rn(hx, s);
  return __fadd2_rn(hs, hs);
}

// Route of one forward element group: 0 SFU tanh, 1 ALU polynomial, 2 ex2.
template <int ACT, int ROUTE>
__device__ __forceinline__ float2 act2_route(float2 hx) {
  if constexpr (ROUTE == 1) return act2_alu<ACT>(hx);
  else if constexpr (ROUTE == 2) return act2_ex2<ACT>(hx);
  else return act2_sfu<ACT>(hx);
}

// act(x) and act'(x) for two lanes from hx = x / 2 (SFU route).
//   GELU: act' = Phi(x) + x phi(x) with Phi(x) ~ s = (1 + t) / 2 (the same
//         tanh as the value) and x phi(x) = x e^(-x^2/2) / sqrt(2 pi)
//         = hx 2^w, w = -2 log2(e) hx^2 + log2(2 / sqrt(2 pi)), from one ex2
//         (the special-function unit has room in the backward, the FMA pipe
//         does not: this takes two fewer packed FMAs than differentiating
//         x s(k(x)), and its error against exact GELU' is smaller, 4.1e-4
//         against 8.7e-4)
//   SiLU: act' = s + x s (1 - s) = s + hx (1 - t^2) / 2
constexpr float kLog2TwoOverSqrt2Pi = -0.3257480647361593f;
template <int ACT>
__device__ __forceinline__ float2 act2_d_sfu(float2 hx, float2& dy) {
  const float2 h2 = __fmul2_rn(hx, hx);
  float2 u = hx;
  if constexpr (ACT == 0) u = __fmul2_rn(hx, __ffma2_rn(h2, f2(4.0f * kGeluB), f2(kGeluA)));
  const float2 t = tanh2_sfu(u);
  const float2 s = __ffma2_rn(t, f2(0.5f), f2(0.5f));
  if constexpr (ACT == 0) {
    const float2 w = __ffma2_rn(h2, f2(-2.0f * kLog2e), f2(kLog2TwoOverSqrt2Pi));
    dy = __ffma2_rn(hx, make_float2(ex2_sfu(w.x), ex2_sfu(w.y)), s);
  } else {
    const float2 q = __ffma2_rn(make_float2(-t.x, -t.y), t, f2(1.0f));
    dy = __ffma2_rn(__fmul2_rn(hx, q), f2(0.5f), s);
  }
  return __ffma2_rn(hx, t, hx);
}
// ALU route: with s = sigmoid(k), s (1 - s) = e s^2 (e = 2^(-k log2 e)):
//   GELU: act' = s (1 + x e s k'(x)),  SiLU: act' = s (1 + x e s)
template <int ACT>
__device__ __forceinline__ float2 act2_d_alu(float2 hx, float2& dy) {
  const float2 h2 = __fmul2_rn(hx, hx);
  float2 w;
  if constexpr (ACT == 0)
    w = __fmul2_rn(hx, __ffma2_rn(h2, f2(-8.0f * kGeluB * kLog2e), f2(-2.0f * kGeluA * kLog2e)));
  else
    w = __fmul2_rn(hx, f2(-2.0f * kLog2e));
  float2 e;
  const float2 s = sigmoid_alu2_w(w, e);
  const float2 x = __fadd2_rn(hx, hx);
  float2 kp;
  if constexpr (ACT == 0) kp = __ffma2_rn(h2, f2(12.0f * kGeluB), f2(kGeluA));  // k'(x) = a + 3 b x^2
  else kp = f2(1.0f);
  const float2 xes = __fmul2_rn(__fmul2_rn(x, e), s);
  dy = __fmul2_rn(s, __ffma2_rn(xes, kp, f2(1.0f)));
  return __fmul2_rn(x, s);
}
template <int ACT, bool ALU>
__device__ __forceinline__ float2 act2_d(float2 hx, float2& dy) {
  if constexpr (ALU) return act2_d_alu<ACT>(hx, dy);
  else return act2_d_sfu<ACT>(hx, dy);
}

// Dispatch on (act, route) at compile time.  ACT: 0 = GELU, 1 = SiLU.
template <int ACT, bool ALU>
__device__ __forceinline__ float act_val(float x) {
  if constexpr (ACT == 0) return ALU ? gelu_alu(x) : gelu_sfu(x);
  else return ALU ? silu_alu(x) : silu_sfu(x);
}
template <int ACT, bool ALU>
__device__ __forceinline__ float act_val_d(float x, float& dy) {
  if constexpr (ACT == 0) return ALU ? gelu_alu_d(x, dy) : gelu_sfu_d(x, dy);
  else return ALU ? silu_alu_d(x, dy) : silu_sfu_d(x, dy);
}

}  // namespace jg
