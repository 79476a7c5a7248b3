// common.cuh -- device helpers shared by the libckv kernels (sm_103a).
//
// Holds the vector load/store wrappers, the bf16 <-> fp32 conversions, the
// status-word helper and -- most importantly -- the per-channel pooling
// arithmetic.  The arithmetic lives here, once, so that every kernel that
// pools a window (C4 prefill, C4 decode, C128 prefill, C128 decode) executes
// the identical sequence of fp32 operations for a given window: a sequence
// compressed in one prefill, in chunks, or token by token through decode
// yields bit-identical rows.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "ckv.h"  // include/ (on the include path)

namespace ckv {

constexpr uint32_t kInvalidU32 = 0xFFFFFFFFu;
constexpr int kMaxBatch = CKV_MAX_BATCH;

// log2(e) rounded to fp32.  exp(x) is evaluated as exp2(x * log2(e)); the
// product is formed by one fused multiply-add against the channel maximum
// (see PoolAcc), so the rounding of -max*log2(e) is common to every entry of a
// window and cancels in the normalised result.
constexpr float kLog2e = 1.44269504088896340736f;

// Programmatic dependent launch.  Every kernel is launched so that it may
// start while its predecessor on the stream is still running: it first does
// work that depends on nothing a predecessor writes, then pdl_wait() (which
// returns once the preceding grid has completed and its memory is visible),
// and it lets its own successor start launching with pdl_release().
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_release() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ void status_or(uint32_t* d_status, uint32_t bits) {
  if (d_status != nullptr) atomicOr(d_status, bits);
}

// ---------------------------------------------------------------- element I/O
template <typename T>
struct Elem;

template <>
struct Elem<float> {
  static constexpr int kBytes = 4;
  __device__ __forceinline__ static float to_f32(float v) { return v; }
};

template <>
struct Elem<__nv_bfloat16> {
  static constexpr int kBytes = 2;
};

__device__ __forceinline__ float bf16lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16hi(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }

// 16-byte loads.  Streamed data (kv_score rows, state rows) bypasses L1 and is
// marked evict-first; the ape bias goes through the read-only path and stays
// cached.
__device__ __forceinline__ uint4 ld_stream16(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ uint4 ld_cached16(const void* p) { return __ldg(reinterpret_cast<const uint4*>(p)); }

__device__ __forceinline__ void st16(void* p, uint4 v) { *reinterpret_cast<uint4*>(p) = v; }

// Unpacks a 16-byte vector into VEC fp32 values (VEC = 8 for bf16, 4 for fp32).
template <typename T>
__device__ __forceinline__ float unpack(const uint4& v, int j);

template <>
__device__ __forceinline__ float unpack<float>(const uint4& v, int j) {
  const uint32_t w = j == 0 ? v.x : j == 1 ? v.y : j == 2 ? v.z : v.w;
  return __uint_as_float(w);
}

template <>
__device__ __forceinline__ float unpack<__nv_bfloat16>(const uint4& v, int j) {
  const uint32_t w = (j >> 1) == 0 ? v.x : (j >> 1) == 1 ? v.y : (j >> 1) == 2 ? v.z : v.w;
  return (j & 1) ? bf16hi(w) : bf16lo(w);
}

// fp32 -> bf16, round to nearest even (cuda_bf16.h intrinsic).
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// Stores VEC fp32 results as TOut at p (VEC*sizeof(TOut) bytes, 8-byte aligned
// at least).
template <typename TOut, int VEC>
__device__ __forceinline__ void store_row_chunk(TOut* p, const float (&r)[VEC]);

template <>
__device__ __forceinline__ void store_row_chunk<float, 8>(float* p, const float (&r)[8]) {
  st16(p, make_uint4(__float_as_uint(r[0]), __float_as_uint(r[1]), __float_as_uint(r[2]), __float_as_uint(r[3])));
  st16(p + 4, make_uint4(__float_as_uint(r[4]), __float_as_uint(r[5]), __float_as_uint(r[6]), __float_as_uint(r[7])));
}
template <>
__device__ __forceinline__ void store_row_chunk<float, 4>(float* p, const float (&r)[4]) {
  st16(p, make_uint4(__float_as_uint(r[0]), __float_as_uint(r[1]), __float_as_uint(r[2]), __float_as_uint(r[3])));
}
template <>
__device__ __forceinline__ void store_row_chunk<__nv_bfloat16, 8>(__nv_bfloat16* p, const float (&r)[8]) {
  st16(p, make_uint4(pack_bf16x2(r[0], r[1]), pack_bf16x2(r[2], r[3]), pack_bf16x2(r[4], r[5]),
                     pack_bf16x2(r[6], r[7])));
}
template <>
__device__ __forceinline__ void store_row_chunk<__nv_bfloat16, 4>(__nv_bfloat16* p, const float (&r)[4]) {
  *reinterpret_cast<uint2*>(p) = make_uint2(pack_bf16x2(r[0], r[1]), pack_bf16x2(r[2], r[3]));
}

template <typename TOut, int VEC>
__device__ __forceinline__ void store_zero_chunk(TOut* p) {
  float z[VEC];
#pragma unroll
  for (int j = 0; j < VEC; ++j) z[j] = 0.0f;
  store_row_chunk<TOut, VEC>(p, z);
}

// ---------------------------------------------------------------- pooling arithmetic
// The canonical per-channel reduction of one window.  For a channel with
// scores s_i = fp32(score_i) + fp32(ape_i) (one rounding, __fadd_rn) and kv_i:
//   M      = max_i s_i                                   (exact)
//   t_i    = fma(s_i, log2e, -(M*log2e))                 (one rounding)
//   e_i    = 2^t_i                                       (ex2.approx.ftz)
//   l_g    = e_i summed in index order within each group of 16 entries
//   a_g    = fma(kv_i, e_i, a) in index order within the group
//   L, A   = balanced pairwise tree over the groups (1 group for C4's 8 entries,
//            8 groups for C128's 128 entries)
//   out    = A / L                                        (IEEE division)
// Every operation is an explicit round-to-nearest intrinsic, so the compiler
// can neither contract nor reorder it.

__device__ __forceinline__ float score_plus_bias(float score, float bias) { return __fadd_rn(score, bias); }

__device__ __forceinline__ float neg_max_log2e(float m) { return __fmul_rn(m, -kLog2e); }

// 2^x by the hardware approximation (ex2.approx.ftz: a few ulp; results below
// 2^-126 flush to zero, which only drops weights under 1e-38 of the largest).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float weight_of(float s, float nml) { return ex2(__fmaf_rn(s, kLog2e, nml)); }

struct PoolAcc {
  float l;
  float a;
  __device__ __forceinline__ void init() {
    l = 0.0f;
    a = 0.0f;
  }
  __device__ __forceinline__ void add(float kv, float e) {
    l = __fadd_rn(l, e);
    a = __fmaf_rn(kv, e, a);
  }
};

__device__ __forceinline__ float finish(float a, float l) { return __fdiv_rn(a, l); }

// The same operations on two channels at once with the packed fp32x2
// instructions of sm_100+ (add.rn.f32x2 / fma.rn.f32x2): each lane is rounded
// exactly like the scalar instruction, so results are bit-identical to the
// scalar forms above and the instruction count per channel drops.
struct F2 {
  uint64_t v;
};

__device__ __forceinline__ F2 f2_pack(float lo, float hi) {
  F2 r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r.v) : "f"(lo), "f"(hi));
  return r;
}

__device__ __forceinline__ void f2_unpack(F2 x, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(x.v));
}

__device__ __forceinline__ F2 f2_add(F2 a, F2 b) {
  F2 r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r.v) : "l"(a.v), "l"(b.v));
  return r;
}

__device__ __forceinline__ F2 f2_fma(F2 a, F2 b, F2 c) {
  F2 r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r.v) : "l"(a.v), "l"(b.v), "l"(c.v));
  return r;
}

// Two bf16 channels (one 32-bit word, low half first) as an fp32 pair.
__device__ __forceinline__ F2 f2_from_bf16x2(uint32_t w) { return f2_pack(bf16lo(w), bf16hi(w)); }

__device__ __forceinline__ F2 score_plus_bias2(F2 score, F2 bias) { return f2_add(score, bias); }

__device__ __forceinline__ F2 weight_of2(F2 s, F2 nml) {
  const F2 t = f2_fma(s, f2_pack(kLog2e, kLog2e), nml);
  float t0, t1;
  f2_unpack(t, t0, t1);
  return f2_pack(ex2(t0), ex2(t1));
}

struct PoolAcc2 {
  F2 l;
  F2 a;
  __device__ __forceinline__ void init() {
    l = f2_pack(0.0f, 0.0f);
    a = f2_pack(0.0f, 0.0f);
  }
  __device__ __forceinline__ void add(F2 kv, F2 e) {
    l = f2_add(l, e);
    a = f2_fma(kv, e, a);
  }
};

// Tree sum of 8 group partials: ((g0+g1)+(g2+g3)) + ((g4+g5)+(g6+g7)).
__device__ __forceinline__ float tree8(const float* v, int stride) {
  const float s01 = __fadd_rn(v[0 * stride], v[1 * stride]);
  const float s23 = __fadd_rn(v[2 * stride], v[3 * stride]);
  const float s45 = __fadd_rn(v[4 * stride], v[5 * stride]);
  const float s67 = __fadd_rn(v[6 * stride], v[7 * stride]);
  return __fadd_rn(__fadd_rn(s01, s23), __fadd_rn(s45, s67));
}

// ---------------------------------------------------------------- misc
__host__ __device__ __forceinline__ bool plan_c_invalid(const ckv_compress_plan_t& p) {
  return p.seq_len == kInvalidU32;
}

__device__ __forceinline__ ckv_compress_plan_t load_plan_c(const ckv_compress_plan_t* p) {
  const uint4 v = __ldg(reinterpret_cast<const uint4*>(p));
  ckv_compress_plan_t r;
  r.seq_len = v.x;
  r.ragged_bl = v.y;
  r.read_page_0 = static_cast<int32_t>(v.z);
  r.read_page_1 = static_cast<int32_t>(v.w);
  return r;
}

__device__ __forceinline__ ckv_decode_plan_t load_plan_d(const ckv_decode_plan_t* p) {
  const uint4 v = __ldg(reinterpret_cast<const uint4*>(p));
  ckv_decode_plan_t r;
  r.seq_len = v.x;
  r.write_loc = static_cast<int32_t>(v.y);
  r.read_page_0 = static_cast<int32_t>(v.z);
  r.read_page_1 = static_cast<int32_t>(v.w);
  return r;
}

__device__ __forceinline__ uint32_t count_or_capacity(const uint32_t* d_counts, int which, uint32_t capacity) {
  if (d_counts == nullptr) return capacity;
  const uint32_t n = __ldg(d_counts + which);
  return n < capacity ? n : capacity;
}

}  // namespace ckv
