// online.cu -- C128 compression through an online state: one slot of
// (m2 | l | a) x head_dim fp32 per request instead of a 128-row page
// (compressor_v2.py _use_online_compress; the online kernels themselves are
// off-page, the recurrence is derived in include/ckv.h).
//
// Both kernels fold tokens with the same per-channel step (online_fold), in
// position order, and keep the state in fp32 between calls, so a sequence
// folded in one prefill, in chunks or token by token gives the same bits.
// Work unit of the prefill: one planner unit (one request's tokens inside one
// 128-group, consecutive rows of the input and of ape); head_dim / 4 threads
// own 4 channels each and walk the unit's tokens in order, fed from a
// shared-memory ring that a producer warp fills with bulk copies (see
// online_prefill_kernel).
#include <algorithm>
#include <atomic>

#include "async_copy.cuh"
#include "common.cuh"
#include "launch.h"

namespace ckv {
namespace {

constexpr int kOnThreads = 256;  // decode
// Prefill ring: kOnStages stages of kOnTok tokens; a stage holds the tokens'
// input rows (kv | score, 2 * head_dim each) followed by their ape rows
// (head_dim each), one bulk copy for each part.  7 x 2 is 42 KB at head_dim
// 512 bf16: five CTAs fit on an SM, and resident CTAs decide the throughput
// (deeper or wider rings that leave room for fewer CTAs are slower).
constexpr int kOnTok = 7;
constexpr int kOnStages = 2;
constexpr int kOnMaxThreads = 1024 / 4 + 32;  // prefill CTA at the largest head_dim: consumers + producer warp

template <typename TIn>
constexpr int prefill_smem_bytes(int hd) {
  return kOnStages * kOnTok * 3 * hd * static_cast<int>(sizeof(TIn));
}

struct OnlineArgs {
  int head_dim;
  int in_dtype;
  int out_dtype;
  float* state;
  uint64_t slots;
  const void* input;
  uint32_t num_q_tokens;  // prefill: input rows; decode: batch
  const void* ape;
  const ckv_online_unit_t* units;
  const ckv_decode_plan_t* plan_d;
  const uint32_t* d_counts;
  uint32_t capacity;  // prefill: capacity_u; decode: batch
  int out_layout;
  uint32_t out_rows;
  void* out;
  uint32_t* d_status;
  // Prefill runs in two passes.  The first unit of a request may load its slot
  // while the request's last unit (another unit, starting at a group start)
  // would store it, so pass 0 folds every unit but leaves those stores out,
  // and pass 1 -- a second launch, after every load -- refolds those last
  // units (their tokens only) and stores their state.
  int pass;
  uint64_t wait_ns;  // limit of the ordinary waits on asynchronous copies
};

// Running softmax of one channel over the tokens of a group so far, kept as
// m2 = fp32(m * log2(e)) for the running maximum m of s, l and a.
struct OnlineState {
  float m2, l, a;

  __device__ __forceinline__ void start(float s, float kv) {
    m2 = __fmul_rn(s, kLog2e);
    l = 1.0f;
    a = kv;
  }
  // With s2 = fp32(s * log2(e)) and w = 2^-|s2 - m2|: a token that raises the
  // maximum rescales the sums by c = w (= exp(m_old - s)) and enters with
  // weight e = 1; any other enters with weight e = w (c = 1).  Then
  // l = l c + e and a = kv e + (a c).  One exponential either way, chosen by
  // selects so that a warp does not diverge.
  __device__ __forceinline__ void fold(float s, float kv) {
    const float s2 = __fmul_rn(s, kLog2e);
    const bool up = s2 > m2;
    const float w = ex2(-fabsf(__fsub_rn(s2, m2)));
    const float c = up ? w : 1.0f, e = up ? 1.0f : w;
    l = __fmaf_rn(l, c, e);
    a = __fmaf_rn(kv, e, __fmul_rn(a, c));
    m2 = up ? s2 : m2;
  }
};

__device__ __forceinline__ F2 f2_mul(F2 a, F2 b) {
  F2 r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r.v) : "l"(a.v), "l"(b.v));
  return r;
}

// OnlineState::fold on two channels with packed fp32x2 arithmetic; lane for
// lane the same operations, so the same bits.
__device__ __forceinline__ void fold2(OnlineState& q0, OnlineState& q1, F2 s, F2 kv) {
  const F2 s2 = f2_mul(s, f2_pack(kLog2e, kLog2e));
  const F2 d = f2_fma(f2_pack(q0.m2, q1.m2), f2_pack(-1.0f, -1.0f), s2);  // s2 - m2, one rounding
  float d0, d1, t0, t1;
  f2_unpack(d, d0, d1);
  f2_unpack(s2, t0, t1);
  const bool u0 = t0 > q0.m2, u1 = t1 > q1.m2;
  const float w0 = ex2(-fabsf(d0)), w1 = ex2(-fabsf(d1));
  const F2 c = f2_pack(u0 ? w0 : 1.0f, u1 ? w1 : 1.0f);
  const F2 e = f2_pack(u0 ? 1.0f : w0, u1 ? 1.0f : w1);
  const F2 l = f2_fma(f2_pack(q0.l, q1.l), c, e);
  const F2 a = f2_fma(kv, e, f2_mul(f2_pack(q0.a, q1.a), c));
  f2_unpack(l, q0.l, q1.l);
  f2_unpack(a, q0.a, q1.a);
  q0.m2 = u0 ? t0 : q0.m2;
  q1.m2 = u1 ? t1 : q1.m2;
}

__device__ __forceinline__ void online_token(OnlineState& st, bool first, float s, float kv) {
  if (first) st.start(s, kv);
  else st.fold(s, kv);
}

// The 4-channel chunk of one staged row: 8 bytes of bf16 or 16 of fp32.
template <typename T>
struct Raw4;
template <>
struct Raw4<float> {
  float4 v;
  __device__ __forceinline__ F2 pair(int h) const { return h == 0 ? f2_pack(v.x, v.y) : f2_pack(v.z, v.w); }
  __device__ __forceinline__ void load(const float* p) { v = *reinterpret_cast<const float4*>(p); }
  __device__ __forceinline__ float get(int j) const { return j == 0 ? v.x : j == 1 ? v.y : j == 2 ? v.z : v.w; }
};
template <>
struct Raw4<__nv_bfloat16> {
  uint2 v;
  __device__ __forceinline__ F2 pair(int h) const { return f2_from_bf16x2(h == 0 ? v.x : v.y); }
  __device__ __forceinline__ void load(const __nv_bfloat16* p) { v = *reinterpret_cast<const uint2*>(p); }
  __device__ __forceinline__ float get(int j) const {
    return j == 0 ? bf16lo(v.x) : j == 1 ? bf16hi(v.x) : j == 2 ? bf16lo(v.y) : bf16hi(v.y);
  }
};

template <typename T>
__device__ __forceinline__ void load_quad(const T* p, float (&v)[4]);

template <>
__device__ __forceinline__ void load_quad<float>(const float* p, float (&v)[4]) {
  const float4 f = __ldg(reinterpret_cast<const float4*>(p));
  v[0] = f.x;
  v[1] = f.y;
  v[2] = f.z;
  v[3] = f.w;
}

template <>
__device__ __forceinline__ void load_quad<__nv_bfloat16>(const __nv_bfloat16* p, float (&v)[4]) {
  const uint2 u = __ldg(reinterpret_cast<const uint2*>(p));
  v[0] = bf16lo(u.x);
  v[1] = bf16hi(u.x);
  v[2] = bf16lo(u.y);
  v[3] = bf16hi(u.y);
}

__device__ __forceinline__ void load_state(const float* st, int hd, int c0, OnlineState (&q)[4]) {
  const float4 m = *reinterpret_cast<const float4*>(st + c0);
  const float4 l = *reinterpret_cast<const float4*>(st + hd + c0);
  const float4 a = *reinterpret_cast<const float4*>(st + 2 * hd + c0);
  q[0] = {m.x, l.x, a.x};
  q[1] = {m.y, l.y, a.y};
  q[2] = {m.z, l.z, a.z};
  q[3] = {m.w, l.w, a.w};
}

__device__ __forceinline__ void store_state(float* st, int hd, int c0, const OnlineState (&q)[4]) {
  *reinterpret_cast<float4*>(st + c0) = make_float4(q[0].m2, q[1].m2, q[2].m2, q[3].m2);
  *reinterpret_cast<float4*>(st + hd + c0) = make_float4(q[0].l, q[1].l, q[2].l, q[3].l);
  *reinterpret_cast<float4*>(st + 2 * hd + c0) = make_float4(q[0].a, q[1].a, q[2].a, q[3].a);
}

template <typename TOut>
__device__ __forceinline__ void store_quad(TOut* p, const float (&r)[4]) {
  store_row_chunk<TOut, 4>(p, r);
}

// A planner unit as the prefill kernel uses it.
struct UnitInfo {
  uint32_t pos0, ragged0, cnt, orow, flags;
  int32_t slot;
  bool late_store;
};

// Decodes unit record `rec` and decides whether this pass runs it: false for
// padding, for units that belong to the other pass and for records that point
// outside the state, the input or the output (those also set `bad`).  The
// producer and the consumers of a CTA call it on the same records, so they
// agree on the sequence of staged tokens.
__device__ __forceinline__ bool unit_runs(const OnlineArgs& a, const uint4& rec, UnitInfo& u, bool& bad) {
  bad = false;
  if (rec.x == kInvalidU32) return false;
  u.pos0 = rec.x;
  u.ragged0 = rec.y & CKV_RAGGED_MASK;
  u.cnt = rec.y >> CKV_UNIT_COUNT_SHIFT;
  u.slot = static_cast<int32_t>(rec.z);
  u.orow = rec.w & CKV_RAGGED_MASK;
  u.flags = rec.w >> CKV_UNIT_FLAGS_SHIFT;
  u.late_store = (u.flags & CKV_UNIT_STORE) && !(u.flags & CKV_UNIT_LOAD) && (u.pos0 % 128) == 0;
  if (a.pass == 1 && !u.late_store) return false;
  bool ok = u.slot >= 0 && static_cast<uint64_t>(u.slot) < a.slots && u.cnt >= 1 && u.cnt <= 128 &&
            u.ragged0 + u.cnt <= a.num_q_tokens && (u.pos0 % 128) + u.cnt <= 128;
  if ((u.flags & CKV_UNIT_EMIT) && a.out_layout != CKV_OUT_TOKEN) ok = ok && u.orow < a.out_rows;
  bad = !ok;
  return ok;
}

__device__ __forceinline__ uint4 load_unit(const OnlineArgs& a, uint32_t k, uint32_t n) {
  return k < n ? __ldg(reinterpret_cast<const uint4*>(a.units + k))
               : make_uint4(kInvalidU32, kInvalidU32, kInvalidU32, kInvalidU32);
}

// One CTA = head_dim / 4 consumer threads (4 channels each) + one producer
// warp, persistent over units blockIdx.x, blockIdx.x + gridDim.x, ...  Lane 0
// of the producer warp streams every unit's tokens, kOnTok per stage, into the
// kOnStages-stage ring: one bulk copy of the tokens' input rows (consecutive
// rows) and one of their ape rows (consecutive rows, since a unit never
// crosses a group), completing the stage's full barrier; the consumers fold
// the stage's tokens in order and release it through its empty barrier (one
// arrival per consumer warp).  Each side reads the next unit's record one unit
// ahead.  Every wait is bounded; on expiry CKV_STATUS_TIMEOUT is set and the
// CTA stops, after the producer has waited (again bounded) for the copies it
// issued.
template <typename TIn, typename TOut, bool kShortWaits>
__global__ __launch_bounds__(kOnMaxThreads) void online_prefill_kernel(const OnlineArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t full_bar[kOnStages];
  __shared__ __align__(8) uint64_t empty_bar[kOnStages];
  __shared__ volatile int abort_flag;
  const int hd = a.head_dim;
  const int tpu = hd / 4;  // consumer threads
  const int t = threadIdx.x;
  const size_t width = 2 * static_cast<size_t>(hd);
  const uint32_t row_bytes = static_cast<uint32_t>(width * sizeof(TIn));
  const uint32_t ape_bytes = static_cast<uint32_t>(hd * sizeof(TIn));
  const uint32_t stage_bytes = kOnTok * (row_bytes + ape_bytes);
  if (t == 0) {
    for (int s = 0; s < kOnStages; ++s) {
      mbar_init(smem_addr(&full_bar[s]), 1);
      mbar_init(smem_addr(&empty_bar[s]), static_cast<uint32_t>(tpu / 32));
    }
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  pdl_wait();  // units, state and input may come from the previous kernels
  pdl_release();
  const uint32_t n = count_or_capacity(a.d_counts, 1, a.capacity);
  const TIn* input = static_cast<const TIn*>(a.input);
  const TIn* ape = static_cast<const TIn*>(a.ape);

  if (t >= tpu) {
    // ---------------- producer (lane 0 of the last warp)
    if (t != tpu) return;
    uint32_t g = 0;
    uint4 rec = load_unit(a, blockIdx.x, n);
    for (uint32_t k = blockIdx.x; k < n && !abort_flag; k += gridDim.x) {
      const uint4 cur = rec;
      rec = load_unit(a, k + gridDim.x, n);
      UnitInfo u;
      bool bad;
      if (!unit_runs(a, cur, u, bad)) continue;
      const TIn* rows = input + static_cast<size_t>(u.ragged0) * width;
      const TIn* arows = ape + static_cast<size_t>(u.pos0 % 128) * hd;
      for (uint32_t j = 0; j < u.cnt; j += kOnTok, ++g) {
        const int stage = static_cast<int>(g % kOnStages);
        if (!wait_for<kShortWaits>(smem_addr(&empty_bar[stage]), ((g / kOnStages) & 1u) ^ 1u, a.wait_ns)) {
          status_or(a.d_status, CKV_STATUS_TIMEOUT);
          abort_flag = 1;
          break;
        }
        if (abort_flag) break;
        const uint32_t ntok = min(static_cast<uint32_t>(kOnTok), u.cnt - j);
        const uint32_t bar = smem_addr(&full_bar[stage]);
        uint8_t* dst = smem + static_cast<size_t>(stage) * stage_bytes;
        mbar_arrive_expect_tx(bar, ntok * (row_bytes + ape_bytes));
        bulk_g2s(smem_addr(dst), rows + j * width, ntok * row_bytes, bar);
        bulk_g2s(smem_addr(dst + kOnTok * row_bytes), arows + static_cast<size_t>(j) * hd, ntok * ape_bytes, bar);
      }
    }
    // the last kOnStages copies issued (each in its own stage) have landed
    // before the CTA can exit
    for (uint32_t h = g > kOnStages ? g - kOnStages : 0u; h < g; ++h)
      mbar_wait_bounded(smem_addr(&full_bar[h % kOnStages]), (h / kOnStages) & 1u, kWaitLimitNs);
    return;
  }

  // ---------------- consumers: thread t owns channels c0 .. c0 + 3
  const int c0 = 4 * t;
  const int lane = t & 31;
  const bool token = a.out_layout == CKV_OUT_TOKEN;
  TOut* out = static_cast<TOut*>(a.out);
  uint32_t g = 0;
  uint4 rec = load_unit(a, blockIdx.x, n);
  for (uint32_t k = blockIdx.x; k < n; k += gridDim.x) {
    const uint4 cur = rec;
    rec = load_unit(a, k + gridDim.x, n);
    UnitInfo u;
    bool bad;
    if (!unit_runs(a, cur, u, bad)) {
      if (bad && c0 == 0 && a.pass == 0) status_or(a.d_status, CKV_STATUS_BAD_INDEX);
      continue;
    }
    const bool emit = u.flags & CKV_UNIT_EMIT;
    float* st = a.state + static_cast<size_t>(u.slot) * 3 * hd;
    OnlineState q[4];
    if (u.flags & CKV_UNIT_LOAD) load_state(st, hd, c0, q);
    bool stop = false;
    for (uint32_t j = 0; j < u.cnt; j += kOnTok, ++g) {
      const int stage = static_cast<int>(g % kOnStages);
      // each thread decides for itself: one that gives up leaves the kernel,
      // and the warp's __syncwarp below waits only for lanes that have not
      // exited (its stage is then never released, so the producer gives up too)
      if (!wait_for<kShortWaits>(smem_addr(&full_bar[stage]), (g / kOnStages) & 1u, a.wait_ns)) {
        status_or(a.d_status, CKV_STATUS_TIMEOUT);
        abort_flag = 1;
        stop = true;
        break;
      }
      const TIn* srow = reinterpret_cast<const TIn*>(smem + static_cast<size_t>(stage) * stage_bytes);
      const TIn* sape = reinterpret_cast<const TIn*>(smem + static_cast<size_t>(stage) * stage_bytes +
                                                      kOnTok * row_bytes);
#pragma unroll
      for (int d = 0; d < kOnTok; ++d) {
        const uint32_t tt = j + d;
        if (tt < u.cnt) {
          Raw4<TIn> kv, sc, bias;
          kv.load(srow + d * width + c0);
          sc.load(srow + d * width + hd + c0);
          bias.load(sape + d * hd + c0);
          // only a unit's first token can start a group (a unit never crosses one)
          if (tt == 0 && u.pos0 % 128 == 0) {
#pragma unroll
            for (int c = 0; c < 4; ++c) q[c].start(score_plus_bias(sc.get(c), bias.get(c)), kv.get(c));
          } else {
            fold2(q[0], q[1], score_plus_bias2(sc.pair(0), bias.pair(0)), kv.pair(0));
            fold2(q[2], q[3], score_plus_bias2(sc.pair(1), bias.pair(1)), kv.pair(1));
          }
          if (a.pass == 0 && token && !(emit && tt + 1 == u.cnt))
            store_zero_chunk<TOut, 4>(out + (static_cast<size_t>(u.ragged0) + tt) * hd + c0);
        }
      }
      // this warp no longer reads the stage
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&empty_bar[stage]));
    }
    if (stop) break;
    if ((u.flags & CKV_UNIT_STORE) && u.late_store == (a.pass == 1)) store_state(st, hd, c0, q);
    if (emit && a.pass == 0) {
      const float r[4] = {finish(q[0].a, q[0].l), finish(q[1].a, q[1].l), finish(q[2].a, q[2].l),
                          finish(q[3].a, q[3].l)};
      const size_t row = token ? static_cast<size_t>(u.ragged0) + u.cnt - 1 : u.orow;
      store_quad<TOut>(out + row * hd + c0, r);
    }
  }
}

template <typename TIn, typename TOut>
__global__ __launch_bounds__(kOnThreads) void online_decode_kernel(const OnlineArgs a) {
  pdl_wait();
  pdl_release();
  const int hd = a.head_dim;
  const int tpu = hd / 4;
  const uint32_t t = blockIdx.x * kOnThreads + threadIdx.x;
  const uint32_t b = t / tpu;
  const int c0 = 4 * static_cast<int>(t % tpu);
  if (b >= a.capacity) return;
  const TIn* input = static_cast<const TIn*>(a.input);
  const TIn* ape = static_cast<const TIn*>(a.ape);
  TOut* out = static_cast<TOut*>(a.out) + static_cast<size_t>(b) * hd + c0;
  const ckv_decode_plan_t P = load_plan_d(a.plan_d + b);
  const float zero[4] = {0.0f, 0.0f, 0.0f, 0.0f};
  if (P.seq_len == kInvalidU32) {
    store_quad<TOut>(out, zero);
    return;
  }
  if (P.seq_len == 0 || P.write_loc < 0 || static_cast<uint64_t>(P.write_loc) >= a.slots) {
    if (c0 == 0) status_or(a.d_status, CKV_STATUS_BAD_INDEX);
    store_quad<TOut>(out, zero);
    return;
  }
  const uint32_t p = P.seq_len - 1;
  const TIn* row = input + static_cast<size_t>(b) * 2 * hd;
  float kv[4], sc[4], bias[4];
  load_quad<TIn>(row + c0, kv);
  load_quad<TIn>(row + hd + c0, sc);
  load_quad<TIn>(ape + static_cast<size_t>(p % 128) * hd + c0, bias);
  float* st = a.state + static_cast<size_t>(P.write_loc) * 3 * hd;
  OnlineState q[4];
  const bool first = p % 128 == 0;
  if (!first) load_state(st, hd, c0, q);
#pragma unroll
  for (int j = 0; j < 4; ++j) online_token(q[j], first, score_plus_bias(sc[j], bias[j]), kv[j]);
  store_state(st, hd, c0, q);
  if ((p + 1) % 128 == 0) {
    const float r[4] = {finish(q[0].a, q[0].l), finish(q[1].a, q[1].l), finish(q[2].a, q[2].l),
                        finish(q[3].a, q[3].l)};
    store_quad<TOut>(out, r);
  } else {
    store_quad<TOut>(out, zero);
  }
}

__global__ void plan_online_decode_kernel(const int64_t* rid, const int64_t* seq_lens, uint32_t batch,
                                          int64_t slot_offset, ckv_decode_plan_t* plan_d, uint32_t* d_status) {
  pdl_wait();
  pdl_release();
  const uint32_t b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= batch) return;
  const int64_t sl = seq_lens[b], r = rid[b];
  uint4 rec = make_uint4(kInvalidU32, kInvalidU32, kInvalidU32, kInvalidU32);
  const int64_t slot = r + slot_offset;
  if (sl >= 1 && sl <= INT32_MAX && r >= 0 && slot >= 0 && slot <= INT32_MAX) {
    const uint32_t s32 = static_cast<uint32_t>(slot);
    rec = make_uint4(static_cast<uint32_t>(sl), s32, s32, s32);
  } else {
    status_or(d_status, CKV_STATUS_BAD_LENGTH);
  }
  *reinterpret_cast<uint4*>(plan_d + b) = rec;
}

int check_online(const OnlineArgs& a) {
  if (a.head_dim <= 0 || a.head_dim % 128 != 0 || a.head_dim > 1024) return CKV_ERR_HEAD_DIM;
  if ((a.in_dtype != CKV_F32 && a.in_dtype != CKV_BF16) || (a.out_dtype != CKV_F32 && a.out_dtype != CKV_BF16) ||
      (a.out_layout != CKV_OUT_TOKEN && a.out_layout != CKV_OUT_COMPACT))
    return CKV_ERR_DTYPE;
  if (a.capacity == 0) return CKV_OK;
  if (!aligned16(a.state) || !aligned16(a.input) || !aligned16(a.ape) || !aligned16(a.out)) return CKV_ERR_POINTER;
  return CKV_OK;
}

// Prefill: head_dim / 4 consumer threads + the producer warp; as many CTAs as
// fit on the GPU at once (at most one per unit).
template <typename TIn, typename TOut, bool kShortWaits>
int launch_prefill(const OnlineArgs& a, cudaStream_t s) {
  auto fn = online_prefill_kernel<TIn, TOut, kShortWaits>;
  const int smem = prefill_smem_bytes<TIn>(a.head_dim);
  const int threads = a.head_dim / 4 + 32;
  // per-device caches (atomics: a repeated set-up by racing threads is harmless)
  static std::atomic<bool> configured[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return CKV_ERR_LAUNCH;
  const bool cached_dev = dev >= 0 && dev < 64;
  if (!cached_dev || !configured[dev].load(std::memory_order_acquire)) {
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, prefill_smem_bytes<TIn>(1024)) !=
        cudaSuccess) {
      cudaGetLastError();
      return CKV_ERR_LAUNCH;
    }
    if (cached_dev) configured[dev].store(true, std::memory_order_release);
  }
  // resident CTAs per SM, per device and head_dim / 128 (the occupancy query is not free on the host)
  static std::atomic<int> per_sm_cache[64][9];
  const int hi = a.head_dim / 128;
  int per_sm = cached_dev ? per_sm_cache[dev][hi].load(std::memory_order_relaxed) : 0;
  if (per_sm == 0) {
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, threads, smem) != cudaSuccess || per_sm < 1) {
      cudaGetLastError();
      return CKV_ERR_LAUNCH;
    }
    if (cached_dev) per_sm_cache[dev][hi].store(per_sm, std::memory_order_relaxed);
  }
  const uint32_t grid = std::max<uint32_t>(
      1, std::min<uint32_t>(a.capacity, static_cast<uint32_t>(per_sm) * static_cast<uint32_t>(sm_count())));
  return launch_pdl(fn, dim3(grid), dim3(threads), smem, s, a);
}

template <typename TIn, typename TOut>
struct PrefillK {
  // kernels built for waits shorter than try_wait's window only for such limits
  static int launch(const OnlineArgs& a, dim3, cudaStream_t s) {
    return a.wait_ns < kShortWaitNs ? launch_prefill<TIn, TOut, true>(a, s) : launch_prefill<TIn, TOut, false>(a, s);
  }
};
template <typename TIn, typename TOut>
struct DecodeK {
  static int launch(const OnlineArgs& a, dim3 grid, cudaStream_t s) {
    return launch_pdl(online_decode_kernel<TIn, TOut>, grid, dim3(kOnThreads), 0, s, a);
  }
};

template <typename KT>
int launch_one(const OnlineArgs& a, dim3 grid, cudaStream_t s) {
  return KT::launch(a, grid, s);
}

template <template <typename, typename> class K>
int launch_typed(const OnlineArgs& a, dim3 grid, cudaStream_t s) {
  if (a.in_dtype == CKV_BF16) {
    if (a.out_dtype == CKV_BF16) return launch_one<K<__nv_bfloat16, __nv_bfloat16>>(a, grid, s);
    return launch_one<K<__nv_bfloat16, float>>(a, grid, s);
  }
  if (a.out_dtype == CKV_BF16) return launch_one<K<float, __nv_bfloat16>>(a, grid, s);
  return launch_one<K<float, float>>(a, grid, s);
}

}  // namespace
}  // namespace ckv

using namespace ckv;

extern "C" int ckv_compress_online_prefill(int head_dim, int in_dtype, int out_dtype, float* state, uint64_t slots,
                                           const void* kv_score_input, uint32_t num_q_tokens, const void* ape,
                                           const ckv_online_unit_t* units, const uint32_t* d_counts,
                                           uint32_t capacity_u, int out_layout, uint32_t out_rows, void* out,
                                           uint32_t* d_status, ckv_stream_t stream) {
  OnlineArgs a{};
  a.head_dim = head_dim;
  a.in_dtype = in_dtype;
  a.out_dtype = out_dtype;
  a.state = state;
  a.slots = slots;
  a.input = kv_score_input;
  a.num_q_tokens = num_q_tokens;
  a.ape = ape;
  a.units = units;
  a.d_counts = d_counts;
  a.capacity = capacity_u;
  a.out_layout = out_layout;
  a.out_rows = out_rows;
  a.out = out;
  a.d_status = d_status;
  a.wait_ns = wait_limit_ns();
  const int rc = check_online(a);
  if (rc || capacity_u == 0) return rc;
  if (!aligned16(units) || (d_counts && (reinterpret_cast<uintptr_t>(d_counts) & 3u))) return CKV_ERR_POINTER;
  a.pass = 0;
  const int rc0 = launch_typed<PrefillK>(a, dim3(1), reinterpret_cast<cudaStream_t>(stream));
  if (rc0) return rc0;
  a.pass = 1;
  return launch_typed<PrefillK>(a, dim3(1), reinterpret_cast<cudaStream_t>(stream));
}

extern "C" int ckv_compress_online_decode(int head_dim, int in_dtype, int out_dtype, float* state, uint64_t slots,
                                          const void* kv_score_input, const void* ape,
                                          const ckv_decode_plan_t* plan_d, uint32_t batch, void* out,
                                          uint32_t* d_status, ckv_stream_t stream) {
  OnlineArgs a{};
  a.head_dim = head_dim;
  a.in_dtype = in_dtype;
  a.out_dtype = out_dtype;
  a.state = state;
  a.slots = slots;
  a.input = kv_score_input;
  a.num_q_tokens = batch;
  a.ape = ape;
  a.plan_d = plan_d;
  a.capacity = batch;
  a.out_layout = CKV_OUT_COMPACT;
  a.out = out;
  a.d_status = d_status;
  const int rc = check_online(a);
  if (rc || batch == 0) return rc;
  if (!aligned16(plan_d)) return CKV_ERR_POINTER;
  const uint64_t threads = static_cast<uint64_t>(batch) * (head_dim / 4);
  const dim3 grid(static_cast<uint32_t>((threads + kOnThreads - 1) / kOnThreads));
  return launch_typed<DecodeK>(a, grid, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" int ckv_plan_online_decode(const int64_t* rid, const int64_t* seq_lens, uint32_t batch,
                                      int64_t slot_offset, ckv_decode_plan_t* plan_d, uint32_t* d_status,
                                      ckv_stream_t stream) {
  if (batch == 0) return CKV_OK;
  if (!rid || !seq_lens || !aligned16(plan_d)) return CKV_ERR_POINTER;
  if ((reinterpret_cast<uintptr_t>(rid) | reinterpret_cast<uintptr_t>(seq_lens)) & 7u) return CKV_ERR_POINTER;
  const uint32_t threads = 256;
  return launch_pdl(plan_online_decode_kernel, dim3((batch + threads - 1) / threads), dim3(threads), 0,
                    reinterpret_cast<cudaStream_t>(stream), rid, seq_lens, batch, slot_offset, plan_d, d_status);
}
