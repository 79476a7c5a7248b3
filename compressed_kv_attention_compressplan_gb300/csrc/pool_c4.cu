// pool_c4.cu -- ratio-4 ("C4") pooling: ragged prefill and fused decode.
//
// C4 rows are | kv-overlap | kv | score-overlap | score | (4 * head_dim).  The
// window of the event ending at position p is positions p-7 .. p: entries
// 0..3 (the previous group) contribute their overlap halves, entries 4..7
// (the current group) their main halves (c4.cuh c4_forward).  An entry comes
// from the request's 8-slot ring when it precedes the extend (i < buffer_len)
// and from the ragged input otherwise.  At seq_len == 4 the previous group
// does not exist and entries 0..3 are left out (c4.cuh sets kv = 0 and
// score = -1e9 there, which gives them weight exactly 0).
//
// Mapping: a "unit" is (event, 16-byte chunk of channels).  A thread owns one
// chunk (8 bf16 or 4 fp32 channels) for the whole grid-stride loop, so the
// ape slice it reads stays in L1; per event it issues 16 independent 16-byte
// loads (kv and score of 8 entries) before any arithmetic.  The window is
// small enough that the fp32 safe softmax runs entirely in registers.
#include <algorithm>

#include "common.cuh"
#include "launch.h"

namespace ckv {
namespace {

constexpr int kC4Threads = 256;

template <typename TIn>
struct C4Vec {
  static constexpr int VEC = 16 / static_cast<int>(sizeof(TIn));  // channels per 16-byte chunk
};

// The C4 window pool for VEC channels.  Entries below `first` are masked.
// (Scalar form: with 16 kv/score vectors live, the packed fp32x2 form of the
// same operations needs more registers than this kernel can spare.)
template <typename TIn, int VEC>
__device__ __forceinline__ void c4_pool_chunk(const uint4 (&kv)[8], const uint4 (&sc)[8], const uint4 (&ap)[8],
                                              int first, float (&res)[VEC]) {
#pragma unroll
  for (int j = 0; j < VEC; ++j) {
    float s[8];
    float m = -INFINITY;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      s[i] = score_plus_bias(unpack<TIn>(sc[i], j), unpack<TIn>(ap[i], j));
      if (i >= first) m = fmaxf(m, s[i]);
    }
    const float nml = neg_max_log2e(m);
    PoolAcc acc;
    acc.init();
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      if (i >= first) acc.add(unpack<TIn>(kv[i], j), weight_of(s[i], nml));
    }
    res[j] = finish(acc.a, acc.l);
  }
}

template <typename TIn, typename TOut>
__global__ __launch_bounds__(kC4Threads, 2) void c4_pool_prefill_kernel(const PoolArgs a, uint32_t chunks,
                                                                     uint32_t units) {
  constexpr int VEC = C4Vec<TIn>::VEC;
  const int hd = a.head_dim;
  const size_t width = 4 * static_cast<size_t>(hd);
  const TIn* state = static_cast<const TIn*>(a.state);
  const TIn* input = static_cast<const TIn*>(a.input);
  const TIn* ape = static_cast<const TIn*>(a.ape);
  TOut* out = static_cast<TOut*>(a.out);
  const bool token = a.out_layout == CKV_OUT_TOKEN;

  pdl_wait();
  pdl_release();
  const uint32_t gid = blockIdx.x * blockDim.x + threadIdx.x;
  const uint32_t stride = gridDim.x * blockDim.x;  // a multiple of `chunks`
  const uint32_t ch = gid % chunks;
  const int c0 = static_cast<int>(ch) * VEC;

  const uint32_t num_c = count_or_capacity(a.d_counts, 0, a.capacity);
  for (uint32_t u = gid; u < units; u += stride) {
    const uint32_t e = u / chunks;
    if (e < num_c) {
      const ckv_compress_plan_t P = load_plan_c(a.plan_c + e);
      if (plan_c_invalid(P)) continue;
      const uint32_t ragged = P.ragged_bl & CKV_RAGGED_MASK;
      const int bl = static_cast<int>(P.ragged_bl >> CKV_BUFFER_LEN_SHIFT);
      const int first = P.seq_len == 4 ? 4 : 0;
      const int64_t rp0 = P.read_page_0, rp1 = P.read_page_1;
      bool ok = ragged < a.num_q_tokens && bl <= 7 && static_cast<int64_t>(ragged) - 7 + bl >= 0;
      if (bl > first && first < 4) ok = ok && rp0 >= 0 && static_cast<uint64_t>(rp0) * 4 + 3 < a.state_rows;
      if (bl > 4) ok = ok && rp1 >= 0 && static_cast<uint64_t>(rp1) * 4 + 3 < a.state_rows;
      if (!ok) {
        if (ch == 0) status_or(a.d_status, CKV_STATUS_BAD_INDEX);
        continue;
      }
      uint4 kv[8], sc[8], ap[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        if (i < first) {
          kv[i] = sc[i] = make_uint4(0, 0, 0, 0);
          continue;
        }
        const TIn* row = i < bl ? state + static_cast<size_t>((i < 4 ? rp0 : rp1) * 4 + (i & 3)) * width
                                : input + (static_cast<size_t>(ragged) + i - 7) * width;
        kv[i] = ld_stream16(row + (i < 4 ? 0 : hd) + c0);
        sc[i] = ld_stream16(row + (i < 4 ? 2 * hd : 3 * hd) + c0);
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) ap[i] = ld_cached16(ape + static_cast<size_t>(i) * hd + c0);  // L1-resident
      float res[VEC];
      c4_pool_chunk<TIn, VEC>(kv, sc, ap, first, res);
      const size_t orow = token ? ragged : e;
      store_row_chunk<TOut, VEC>(out + orow * hd + c0, res);
      if (token) {
        // zero the rows between the previous compress row and this one
        int64_t prev = -1;
        if (e > 0) {
          const ckv_compress_plan_t Q = load_plan_c(a.plan_c + e - 1);
          prev = plan_c_invalid(Q) ? static_cast<int64_t>(ragged) : static_cast<int64_t>(Q.ragged_bl & CKV_RAGGED_MASK);
        }
        for (int64_t r = prev + 1; r < static_cast<int64_t>(ragged); ++r)
          store_zero_chunk<TOut, VEC>(out + static_cast<size_t>(r) * hd + c0);
      }
    } else if (token && e == num_c) {
      // rows after the last compress row
      int64_t last = -1;
      if (num_c > 0) {
        const ckv_compress_plan_t Q = load_plan_c(a.plan_c + num_c - 1);
        last = plan_c_invalid(Q) ? static_cast<int64_t>(a.num_q_tokens) : static_cast<int64_t>(Q.ragged_bl & CKV_RAGGED_MASK);
      }
      for (int64_t r = last + 1; r < static_cast<int64_t>(a.num_q_tokens); ++r)
        store_zero_chunk<TOut, VEC>(out + static_cast<size_t>(r) * hd + c0);
    }
  }
}

// Decode: one unit per (row, chunk).  The new token's row is written to its
// ring slot; at a group boundary the window's first 7 entries come from the
// ring (none of them is the slot being written) and entry 7 is the new token.
// The new token's chunk and the ape chunks do not depend on the plan record,
// so they are requested together with it: a boundary row costs two memory
// round trips (record + token + ape, then the ring rows), any other row one.
constexpr int kC4DecodeThreads = 128;  // 128-thread blocks: a batch of 256 rows x 64 chunks covers every SM

template <typename TIn, typename TOut>
__global__ __launch_bounds__(kC4DecodeThreads) void c4_decode_kernel(const PoolArgs a, uint32_t chunks,
                                                                     uint32_t units) {
  constexpr int VEC = C4Vec<TIn>::VEC;
  pdl_wait();
  pdl_release();
  const uint32_t u = blockIdx.x * blockDim.x + threadIdx.x;
  if (u >= units) return;
  const int hd = a.head_dim;
  const size_t width = 4 * static_cast<size_t>(hd);
  TIn* state = static_cast<TIn*>(a.state_mut);
  const TIn* input = static_cast<const TIn*>(a.input);
  const TIn* ape = static_cast<const TIn*>(a.ape);
  TOut* out = static_cast<TOut*>(a.out);
  const uint32_t b = u / chunks;
  const uint32_t ch = u % chunks;
  const int c0 = static_cast<int>(ch) * VEC;
  TOut* orow = out + static_cast<size_t>(b) * hd + c0;

  const ckv_decode_plan_t P = load_plan_d(a.plan_d + b);
  const TIn* src = input + static_cast<size_t>(b) * width + c0;  // row b of the input always exists
  const uint4 kv_ovl = ld_stream16(src), kv_main = ld_stream16(src + hd);
  const uint4 sc_ovl = ld_stream16(src + 2 * hd), sc_main = ld_stream16(src + 3 * hd);
  uint4 ap[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) ap[i] = ld_cached16(ape + static_cast<size_t>(i) * hd + c0);
  if (P.seq_len == kInvalidU32) {
    store_zero_chunk<TOut, VEC>(orow);
    return;
  }
  const bool boundary = P.seq_len % 4 == 0;
  const int64_t rp0 = P.read_page_0, rp1 = P.read_page_1;
  bool ok = P.write_loc >= 0 && static_cast<uint64_t>(P.write_loc) < a.state_rows;
  if (boundary)
    ok = ok && rp0 >= 0 && rp1 >= 0 && static_cast<uint64_t>(rp0) * 4 + 3 < a.state_rows &&
         static_cast<uint64_t>(rp1) * 4 + 3 < a.state_rows;
  if (!ok) {
    if (ch == 0) status_or(a.d_status, CKV_STATUS_BAD_INDEX);
    store_zero_chunk<TOut, VEC>(orow);
    return;
  }
  TIn* dst = state + static_cast<size_t>(P.write_loc) * width + c0;
  st16(dst, kv_ovl);
  st16(dst + hd, kv_main);
  st16(dst + 2 * hd, sc_ovl);
  st16(dst + 3 * hd, sc_main);
  if (!boundary) {
    store_zero_chunk<TOut, VEC>(orow);
    return;
  }
  const int first = P.seq_len == 4 ? 4 : 0;
  uint4 kv[8], sc[8];
#pragma unroll
  for (int i = 0; i < 7; ++i) {
    if (i < first) {
      kv[i] = sc[i] = make_uint4(0, 0, 0, 0);
      continue;
    }
    const TIn* row = state + static_cast<size_t>((i < 4 ? rp0 : rp1) * 4 + (i & 3)) * width;
    kv[i] = ld_stream16(row + (i < 4 ? 0 : hd) + c0);
    sc[i] = ld_stream16(row + (i < 4 ? 2 * hd : 3 * hd) + c0);
  }
  kv[7] = kv_main;
  sc[7] = sc_main;
  float res[VEC];
  c4_pool_chunk<TIn, VEC>(kv, sc, ap, first, res);
  store_row_chunk<TOut, VEC>(orow, res);
}

template <typename TIn, typename TOut>
int launch_prefill_t(const PoolArgs& a, cudaStream_t s) {
  constexpr int VEC = C4Vec<TIn>::VEC;
  const uint32_t chunks = static_cast<uint32_t>(a.head_dim / VEC);
  const uint32_t threads = (kC4Threads / chunks) * chunks;
  const uint64_t units64 =
      (static_cast<uint64_t>(a.capacity) + (a.out_layout == CKV_OUT_TOKEN ? 1 : 0)) * chunks;
  if (units64 == 0) return CKV_OK;
  if (units64 > 0xFFFFFFFFull) return CKV_ERR_SIZE;
  const uint32_t units = static_cast<uint32_t>(units64);
  uint32_t grid = (units + threads - 1) / threads;
  grid = std::max<uint32_t>(1, std::min<uint32_t>(grid, 16u * static_cast<uint32_t>(sm_count())));
  return launch_pdl(c4_pool_prefill_kernel<TIn, TOut>, dim3(grid), dim3(threads), 0, s, a, chunks, units);
}

template <typename TIn, typename TOut>
int launch_decode_t(const PoolArgs& a, cudaStream_t s) {
  constexpr int VEC = C4Vec<TIn>::VEC;
  const uint32_t chunks = static_cast<uint32_t>(a.head_dim / VEC);
  const uint64_t units64 = static_cast<uint64_t>(a.capacity) * chunks;
  if (units64 == 0) return CKV_OK;
  if (units64 > 0xFFFFFFFFull) return CKV_ERR_SIZE;
  const uint32_t units = static_cast<uint32_t>(units64);
  constexpr uint32_t threads = kC4DecodeThreads;
  return launch_pdl(c4_decode_kernel<TIn, TOut>, dim3((units + threads - 1) / threads), dim3(threads), 0, s, a,
                    chunks, units);
}

}  // namespace

int launch_c4_pool_prefill(const PoolArgs& a, cudaStream_t s) {
  if (a.in_dtype == CKV_BF16)
    return a.out_dtype == CKV_BF16 ? launch_prefill_t<__nv_bfloat16, __nv_bfloat16>(a, s)
                                   : launch_prefill_t<__nv_bfloat16, float>(a, s);
  return a.out_dtype == CKV_BF16 ? launch_prefill_t<float, __nv_bfloat16>(a, s) : launch_prefill_t<float, float>(a, s);
}

int launch_c4_decode(const PoolArgs& a, cudaStream_t s) {
  if (a.in_dtype == CKV_BF16)
    return a.out_dtype == CKV_BF16 ? launch_decode_t<__nv_bfloat16, __nv_bfloat16>(a, s)
                                   : launch_decode_t<__nv_bfloat16, float>(a, s);
  return a.out_dtype == CKV_BF16 ? launch_decode_t<float, __nv_bfloat16>(a, s) : launch_decode_t<float, float>(a, s);
}

}  // namespace ckv
