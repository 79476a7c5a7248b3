// pool_c128.cu -- ratio-128 ("C128") pooling: ragged prefill and fused decode.
//
// C128 rows are | kv | score | (2 * head_dim).  The window of the event ending
// at position p is positions p-127 .. p, i.e. the whole 128-slot page of the
// request (compressor_v2.py _compress_forward_c128_fallback: softmax of
// score + ape over the 128 slots, weighted sum of kv).  Entry i comes from the
// page (slot i) when it precedes the extend (i < buffer_len) and from ragged
// input row ragged_id - 127 + i otherwise; in decode entries 0..126 come from
// the page and entry 127 is the new token.
//
// Mapping: one CTA per tile = (event, slice of CS channels).  The tile's 128
// entries x CS channels of kv and of score (64 KB) are staged in shared
// memory by 256 one-dimensional bulk copies (cp.async.bulk, the TMA engine)
// that all signal one mbarrier, so every byte of the tile is in flight at once
// and no register holds staged data.  The arithmetic then reads shared memory:
// 8 groups of 16 consecutive entries x CS/4 channel quads; pass 1 forms the
// scores and the exact per-channel maximum, pass 2 the group sums of weights
// and weighted kv, pass 3 the fixed pairwise tree over the 8 groups.
#include <algorithm>

#include "common.cuh"
#include "launch.h"

namespace ckv {
namespace {

template <typename TIn>
struct C128Cfg {
  static constexpr int CS = sizeof(TIn) == 2 ? 128 : 64;          // channels per tile
  static constexpr int QUADS = CS / 4;                            // 4 channels per thread
  static constexpr int THREADS = QUADS * 8;                       // 8 entry groups
  static constexpr int SEG_BYTES = CS * static_cast<int>(sizeof(TIn));  // one entry's kv (or score) slice
  static constexpr int TILE_BYTES = 128 * SEG_BYTES * 2;          // 64 KB
  static constexpr int RED_BYTES = 2 * 8 * CS * 4;                // group partials (l, a)
  static constexpr int SMEM_BYTES = TILE_BYTES + RED_BYTES;
};

// ---------------------------------------------------------------- TMA / mbarrier
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Waits for phase `parity` of the barrier for at most `limit_ns` nanoseconds.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (global_ns() - t0 > limit_ns) return false;
  }
}

// One bulk global -> shared copy that completes `bytes` of the barrier's
// transaction count.  dst and src 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s: far beyond any real copy

// 4 consecutive channels of a staged entry / of ape as fp32.
template <typename TIn>
__device__ __forceinline__ void load4(const TIn* p, float (&v)[4]);

template <>
__device__ __forceinline__ void load4<__nv_bfloat16>(const __nv_bfloat16* p, float (&v)[4]) {
  const uint2 u = *reinterpret_cast<const uint2*>(p);
  v[0] = bf16lo(u.x);
  v[1] = bf16hi(u.x);
  v[2] = bf16lo(u.y);
  v[3] = bf16hi(u.y);
}

template <>
__device__ __forceinline__ void load4<float>(const float* p, float (&v)[4]) {
  const float4 u = *reinterpret_cast<const float4*>(p);
  v[0] = u.x;
  v[1] = u.y;
  v[2] = u.z;
  v[3] = u.w;
}

template <typename TIn>
__device__ __forceinline__ void ldg4(const TIn* p, float (&v)[4]);

template <>
__device__ __forceinline__ void ldg4<__nv_bfloat16>(const __nv_bfloat16* p, float (&v)[4]) {
  const uint2 u = __ldg(reinterpret_cast<const uint2*>(p));
  v[0] = bf16lo(u.x);
  v[1] = bf16hi(u.x);
  v[2] = bf16lo(u.y);
  v[3] = bf16hi(u.y);
}

template <>
__device__ __forceinline__ void ldg4<float>(const float* p, float (&v)[4]) {
  const float4 u = __ldg(reinterpret_cast<const float4*>(p));
  v[0] = u.x;
  v[1] = u.y;
  v[2] = u.z;
  v[3] = u.w;
}

template <typename TOut>
__device__ __forceinline__ void store1(TOut* p, float v);
template <>
__device__ __forceinline__ void store1<float>(float* p, float v) {
  *p = v;
}
template <>
__device__ __forceinline__ void store1<__nv_bfloat16>(__nv_bfloat16* p, float v) {
  *p = __float2bfloat16_rn(v);
}

// Zero rows [r0, r1) of out, columns [c0, c0 + CS).
template <typename TIn, typename TOut>
__device__ __forceinline__ void zero_rows(TOut* out, int hd, int c0, int64_t r0, int64_t r1) {
  using Cfg = C128Cfg<TIn>;
  constexpr int kPerRow = Cfg::CS * static_cast<int>(sizeof(TOut)) / 16;
  constexpr int kElems = 16 / static_cast<int>(sizeof(TOut));
  const int64_t total = (r1 - r0) * kPerRow;
  for (int64_t idx = threadIdx.x; idx < total; idx += Cfg::THREADS) {
    const int64_t r = r0 + idx / kPerRow;
    const int c = c0 + static_cast<int>(idx % kPerRow) * kElems;
    st16(out + r * hd + c, make_uint4(0, 0, 0, 0));
  }
}

// The C128 pooling kernel.  kDecode: tiles are (batch row, slice) of a decode
// step; otherwise (compress record, slice) of a prefill step.
template <typename TIn, typename TOut, bool kDecode>
__global__ __launch_bounds__(C128Cfg<TIn>::THREADS, 2) void c128_pool_kernel(const PoolArgs a, uint32_t slices,
                                                                               uint32_t tiles) {
  using Cfg = C128Cfg<TIn>;
  constexpr int CS = Cfg::CS;
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t bar_storage;
  TIn* kv_s = reinterpret_cast<TIn*>(smem);
  TIn* sc_s = kv_s + 128 * CS;
  float* red_l = reinterpret_cast<float*>(smem + Cfg::TILE_BYTES);
  float* red_a = red_l + 8 * CS;

  const uint32_t tile = blockIdx.x;
  if (tile >= tiles) return;
  const uint32_t e = tile / slices;
  const int c0 = static_cast<int>(tile % slices) * CS;
  const int hd = a.head_dim;
  const size_t width = 2 * static_cast<size_t>(hd);
  const int t = threadIdx.x;
  const TIn* input = static_cast<const TIn*>(a.input);
  const TIn* state = kDecode ? static_cast<const TIn*>(a.state_mut) : static_cast<const TIn*>(a.state);
  TOut* out = static_cast<TOut*>(a.out);

  uint32_t ragged;
  int bl;
  int64_t rp0;
  size_t orow;
  if constexpr (kDecode) {
    const ckv_decode_plan_t P = load_plan_d(a.plan_d + e);
    orow = e;
    if (P.seq_len == kInvalidU32) {
      zero_rows<TIn, TOut>(out, hd, c0, e, e + 1);
      return;
    }
    const bool boundary = P.seq_len % 128 == 0;
    rp0 = P.read_page_0;
    bool ok = P.write_loc >= 0 && static_cast<uint64_t>(P.write_loc) < a.state_rows;
    if (boundary) ok = ok && rp0 >= 0 && static_cast<uint64_t>(rp0) * 128 + 127 < a.state_rows;
    if (!ok) {
      if (t == 0) status_or(a.d_status, CKV_STATUS_BAD_INDEX);
      zero_rows<TIn, TOut>(out, hd, c0, e, e + 1);
      return;
    }
    // the new token's slice of kv and score goes to its page slot
    if (t < 2 * Cfg::SEG_BYTES / 16) {
      const int half = t / (Cfg::SEG_BYTES / 16);
      const int off = (t % (Cfg::SEG_BYTES / 16)) * (16 / static_cast<int>(sizeof(TIn)));
      const TIn* src = input + static_cast<size_t>(e) * width + half * hd + c0 + off;
      TIn* dst = static_cast<TIn*>(a.state_mut) + static_cast<size_t>(P.write_loc) * width + half * hd + c0 + off;
      st16(dst, ld_stream16(src));
    }
    if (!boundary) {
      zero_rows<TIn, TOut>(out, hd, c0, e, e + 1);
      return;
    }
    ragged = e;
    bl = 127;
  } else {
    const uint32_t num_c = count_or_capacity(a.d_counts, 0, a.capacity);
    const bool token = a.out_layout == CKV_OUT_TOKEN;
    if (e >= num_c) {
      if (token && e == num_c) {  // rows after the last compress row
        int64_t last = -1;
        if (num_c > 0) {
          const ckv_compress_plan_t Q = load_plan_c(a.plan_c + num_c - 1);
          last = plan_c_invalid(Q) ? static_cast<int64_t>(a.num_q_tokens)
                                   : static_cast<int64_t>(Q.ragged_bl & CKV_RAGGED_MASK);
        }
        zero_rows<TIn, TOut>(out, hd, c0, last + 1, a.num_q_tokens);
      }
      return;
    }
    const ckv_compress_plan_t P = load_plan_c(a.plan_c + e);
    if (plan_c_invalid(P)) return;
    ragged = P.ragged_bl & CKV_RAGGED_MASK;
    bl = static_cast<int>(P.ragged_bl >> CKV_BUFFER_LEN_SHIFT);
    rp0 = P.read_page_0;
    bool ok = ragged < a.num_q_tokens && bl <= 127 && static_cast<int64_t>(ragged) - 127 + bl >= 0;
    if (bl > 0) ok = ok && rp0 >= 0 && static_cast<uint64_t>(rp0) * 128 + 127 < a.state_rows;
    if (!ok) {
      if (t == 0) status_or(a.d_status, CKV_STATUS_BAD_INDEX);
      return;
    }
    orow = token ? ragged : e;
    if (token) {  // rows between the previous compress row and this one
      int64_t prev = -1;
      if (e > 0) {
        const ckv_compress_plan_t Q = load_plan_c(a.plan_c + e - 1);
        prev = plan_c_invalid(Q) ? static_cast<int64_t>(ragged) : static_cast<int64_t>(Q.ragged_bl & CKV_RAGGED_MASK);
      }
      zero_rows<TIn, TOut>(out, hd, c0, prev + 1, ragged);
    }
  }

  // ---- stage the tile: 128 entries x (kv slice, score slice)
  const uint32_t bar = smem_addr(&bar_storage);
  if (t == 0) mbar_init(bar, 1);
  __syncthreads();
  if (t < 32) {
    if (t == 0) mbar_arrive_expect_tx(bar, Cfg::TILE_BYTES);
    __syncwarp();
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int i = t + 32 * k;
      const TIn* row = i < bl ? state + (static_cast<size_t>(rp0) * 128 + i) * width
                              : input + (static_cast<size_t>(ragged) + i - 127) * width;
      bulk_g2s(smem_addr(kv_s + i * CS), row + c0, Cfg::SEG_BYTES, bar);
      bulk_g2s(smem_addr(sc_s + i * CS), row + hd + c0, Cfg::SEG_BYTES, bar);
    }
  }
  if (!mbar_wait_bounded(bar, 0, kWaitLimitNs)) {
    status_or(a.d_status, CKV_STATUS_TIMEOUT);
    mbar_wait_bounded(bar, 0, kWaitLimitNs);  // let copies in flight land before the CTA can exit
  }

  // ---- pass 1: scores and the per-channel maximum
  const int q = t % Cfg::QUADS;
  const int g = t / Cfg::QUADS;
  const int cq = 4 * q;
  const TIn* ape = static_cast<const TIn*>(a.ape) + c0 + cq;
  float s[16][4];
  float m[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
  for (int k = 0; k < 16; ++k) {
    const int i = 16 * g + k;
    float sc[4], bias[4];
    load4<TIn>(sc_s + i * CS + cq, sc);
    ldg4<TIn>(ape + static_cast<size_t>(i) * hd, bias);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      s[k][j] = score_plus_bias(sc[j], bias[j]);
      m[j] = fmaxf(m[j], s[k][j]);
    }
  }
  *reinterpret_cast<float4*>(red_l + g * CS + cq) = make_float4(m[0], m[1], m[2], m[3]);
  __syncthreads();
  float nml[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    float mm = red_l[cq + j];
#pragma unroll
    for (int gg = 1; gg < 8; ++gg) mm = fmaxf(mm, red_l[gg * CS + cq + j]);
    nml[j] = neg_max_log2e(mm);
  }
  __syncthreads();

  // ---- pass 2: group sums of weights and of weighted kv
  PoolAcc acc[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) acc[j].init();
#pragma unroll
  for (int k = 0; k < 16; ++k) {
    const int i = 16 * g + k;
    float kv[4];
    load4<TIn>(kv_s + i * CS + cq, kv);
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[j].add(kv[j], weight_of(s[k][j], nml[j]));
  }
  *reinterpret_cast<float4*>(red_l + g * CS + cq) = make_float4(acc[0].l, acc[1].l, acc[2].l, acc[3].l);
  *reinterpret_cast<float4*>(red_a + g * CS + cq) = make_float4(acc[0].a, acc[1].a, acc[2].a, acc[3].a);
  __syncthreads();

  // ---- pass 3: tree over the 8 groups, one channel per thread
  if (t < CS) {
    const float L = tree8(red_l + t, CS);
    const float A = tree8(red_a + t, CS);
    store1<TOut>(out + orow * hd + c0 + t, finish(A, L));
  }
}

template <typename TIn, typename TOut, bool kDecode>
int launch_t(const PoolArgs& a, cudaStream_t s) {
  using Cfg = C128Cfg<TIn>;
  const uint32_t slices = static_cast<uint32_t>(a.head_dim / Cfg::CS);
  const uint64_t items = kDecode ? a.capacity
                                 : static_cast<uint64_t>(a.capacity) + (a.out_layout == CKV_OUT_TOKEN ? 1 : 0);
  const uint64_t tiles64 = items * slices;
  if (tiles64 == 0) return CKV_OK;
  if (tiles64 > 0x7FFFFFFFull) return CKV_ERR_SIZE;
  // The dynamic shared-memory opt-in is a per-device function attribute.
  static bool configured[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return CKV_ERR_LAUNCH;
  if (dev < 0 || dev >= 64 || !configured[dev]) {
    if (cudaFuncSetAttribute(c128_pool_kernel<TIn, TOut, kDecode>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             Cfg::SMEM_BYTES) != cudaSuccess)
      return CKV_ERR_LAUNCH;
    if (dev >= 0 && dev < 64) configured[dev] = true;
  }
  const uint32_t tiles = static_cast<uint32_t>(tiles64);
  c128_pool_kernel<TIn, TOut, kDecode><<<tiles, Cfg::THREADS, Cfg::SMEM_BYTES, s>>>(a, slices, tiles);
  return check_launch();
}

template <bool kDecode>
int dispatch(const PoolArgs& a, cudaStream_t s) {
  if (a.in_dtype == CKV_BF16)
    return a.out_dtype == CKV_BF16 ? launch_t<__nv_bfloat16, __nv_bfloat16, kDecode>(a, s)
                                   : launch_t<__nv_bfloat16, float, kDecode>(a, s);
  return a.out_dtype == CKV_BF16 ? launch_t<float, __nv_bfloat16, kDecode>(a, s)
                                 : launch_t<float, float, kDecode>(a, s);
}

}  // namespace

int launch_c128_pool_prefill(const PoolArgs& a, cudaStream_t s) { return dispatch<false>(a, s); }
int launch_c128_decode(const PoolArgs& a, cudaStream_t s) { return dispatch<true>(a, s); }

}  // namespace ckv
