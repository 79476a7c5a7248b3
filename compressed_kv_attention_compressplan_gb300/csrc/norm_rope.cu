// norm_rope.cu -- RMSNorm + RoPE + store of the compressed rows into the KV
// cache (compressor_v2.py compress_norm_rope_store, the step after pooling).
//
// Per record: x = the pooled row (zero for a decode row off a ratio boundary),
// y_c = x_c * w_c / sqrt(mean(x^2) + eps), then the last rope_dim channels
// turn as interleaved pairs (2i, 2i+1) by the cos / sin of table row
// pos = max(seq_len - ratio, 0), and y goes to cache row out_loc.  One warp
// owns one record: lane l holds channels 128 j + 4 l .. +3 of every 128-wide
// chunk j, so each rotated pair sits in one lane; the sum of squares is a
// lane-sequential sum followed by a fixed butterfly over the warp.
#include <algorithm>
#include <atomic>

#include <cuda_bf16.h>

#include "common.cuh"
#include "launch.h"

namespace ckv {
namespace {

// Four warps per block: the resident wave then holds more warps than with
// eight (7.32 -> 6.92 us back to back on the C128 prefill rows, 1.92 -> 1.88
// us on the decode rows), and a 512-row decode spreads over 128 SMs, not 64.
constexpr int kNrThreads = 128;

struct NormRopeArgs {
  int ratio;
  int decode;  // 1: plan_d rows (every row stored); 0: plan_c records
  int head_dim;
  int rope_dim;
  int in_dtype;
  int in_layout;
  const void* rows;
  uint64_t n_rows;
  const ckv_compress_plan_t* plan_c;
  const ckv_decode_plan_t* plan_d;
  const uint32_t* d_counts;
  uint32_t capacity;
  const float* weight;
  float eps;
  const float* freqs;
  uint32_t max_pos;
  const int64_t* out_loc;
  uint64_t n_loc;
  int cache_dtype;
  void* cache;
  uint64_t cache_rows;
  uint32_t* d_status;
};

__device__ __forceinline__ void load_chunk(const void* rows, int dtype, size_t idx, float (&v)[4]) {
  if (dtype == CKV_BF16) {
    const uint2 u = __ldg(reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(rows) + idx));
    v[0] = __uint_as_float(u.x << 16);
    v[1] = __uint_as_float(u.x & 0xFFFF0000u);
    v[2] = __uint_as_float(u.y << 16);
    v[3] = __uint_as_float(u.y & 0xFFFF0000u);
  } else {
    const float4 f = __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(rows) + idx));
    v[0] = f.x;
    v[1] = f.y;
    v[2] = f.z;
    v[3] = f.w;
  }
}

__device__ __forceinline__ void store_chunk(void* cache, int dtype, size_t idx, const float (&v)[4]) {
  if (dtype == CKV_BF16) {
    const __nv_bfloat162 lo = __floats2bfloat162_rn(v[0], v[1]);
    const __nv_bfloat162 hi = __floats2bfloat162_rn(v[2], v[3]);
    uint2 u;
    u.x = *reinterpret_cast<const uint32_t*>(&lo);
    u.y = *reinterpret_cast<const uint32_t*>(&hi);
    *reinterpret_cast<uint2*>(static_cast<uint16_t*>(cache) + idx) = u;
  } else {
    *reinterpret_cast<float4*>(static_cast<float*>(cache) + idx) = make_float4(v[0], v[1], v[2], v[3]);
  }
}

// kChunks = head_dim / 128 (1 .. 8): a lane's registers hold exactly its channels.
template <int kChunks>
__global__ __launch_bounds__(kNrThreads) void norm_rope_store_kernel(const NormRopeArgs a) {
  pdl_wait();  // the pooled rows come from the previous kernel
  pdl_release();
  const int lane = threadIdx.x & 31;
  const uint32_t warps_total = gridDim.x * (kNrThreads / 32);
  const uint32_t n = a.decode ? a.capacity : count_or_capacity(a.d_counts, 0, a.capacity);
  const int hd = 128 * kChunks;
  const int base = hd - a.rope_dim;
  const int half = a.rope_dim / 2;
  // Each warp walks records k, k + warps_total, ...; the next record's plan
  // entry is requested before the current record's data, so a record costs
  // one memory round trip once the loop runs.
  const uint4* plan = a.decode ? reinterpret_cast<const uint4*>(a.plan_d) : reinterpret_cast<const uint4*>(a.plan_c);
  const uint4 kNone = make_uint4(kInvalidU32, kInvalidU32, kInvalidU32, kInvalidU32);
  uint32_t k = blockIdx.x * (kNrThreads / 32) + (threadIdx.x >> 5);
  uint4 rec = k < n ? __ldg(plan + k) : kNone;
  for (; k < n; k += warps_total) {
    const uint32_t kn = k + warps_total;
    const uint4 cur = rec;
    rec = kn < n ? __ldg(plan + kn) : kNone;
    if (cur.x == kInvalidU32) continue;  // an invalid record (both kinds start with seq_len)
    uint64_t row, loc_index;
    int64_t pos;
    bool zero = false;
    const uint32_t seq_len = cur.x;
    if (a.decode) {
      row = k;
      loc_index = k;
      zero = seq_len % static_cast<uint32_t>(a.ratio) != 0;
      pos = max(static_cast<int64_t>(seq_len) - a.ratio, int64_t{0});
    } else {
      const uint32_t ragged = cur.y & CKV_RAGGED_MASK;
      row = a.in_layout == CKV_OUT_COMPACT ? k : ragged;
      loc_index = ragged;
      pos = static_cast<int64_t>(seq_len) - a.ratio;
    }
    // everything the record needs is requested at once (one memory round trip
    // after the plan record): its row, its cache location, its table row and
    // the weight; the bounds decide afterwards what is stored
    const bool row_ok = row < a.n_rows;
    const bool pos_ok = pos >= 0 && (a.rope_dim == 0 || pos < a.max_pos);
    const int64_t loc = loc_index < a.n_loc ? __ldg(a.out_loc + loc_index) : -1;
    float v[kChunks][4];
    float4 w[kChunks], cs[kChunks];
#pragma unroll
    for (int j = 0; j < kChunks; ++j) {
      {
        const int c0 = 128 * j + 4 * lane;
        if (zero || !row_ok) {
          v[j][0] = v[j][1] = v[j][2] = v[j][3] = 0.0f;
        } else {
          load_chunk(a.rows, a.in_dtype, row * hd + c0, v[j]);
        }
        w[j] = __ldg(reinterpret_cast<const float4*>(a.weight + c0));
        if (c0 >= base && pos_ok) {  // (cos, sin) of pairs (c0 - base) / 2 and the next one
          const size_t f = (static_cast<size_t>(pos) * half + (c0 - base) / 2) * 2;
          cs[j] = __ldg(reinterpret_cast<const float4*>(a.freqs + f));
        } else {
          cs[j] = make_float4(1.0f, 0.0f, 1.0f, 0.0f);
        }
      }
    }
    if (!row_ok || !pos_ok || loc < 0 || static_cast<uint64_t>(loc) >= a.cache_rows) {
      if (lane == 0) status_or(a.d_status, CKV_STATUS_BAD_INDEX);
      continue;
    }
    float ss = 0.0f;
#pragma unroll
    for (int j = 0; j < kChunks; ++j) {
      {
#pragma unroll
        for (int e = 0; e < 4; ++e) ss = fmaf(v[j][e], v[j][e], ss);
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xFFFFFFFFu, ss, off);
    const float r = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(ss, static_cast<float>(hd)), a.eps)));
#pragma unroll
    for (int j = 0; j < kChunks; ++j) {
      {
        const int c0 = 128 * j + 4 * lane;
        float y[4] = {v[j][0] * r * w[j].x, v[j][1] * r * w[j].y, v[j][2] * r * w[j].z, v[j][3] * r * w[j].w};
        if (c0 >= base) {  // a rotated chunk: pairs (c0, c0+1) and (c0+2, c0+3)
          const float a0 = y[0], b0 = y[1], a1 = y[2], b1 = y[3];
          y[0] = a0 * cs[j].x - b0 * cs[j].y;
          y[1] = a0 * cs[j].y + b0 * cs[j].x;
          y[2] = a1 * cs[j].z - b1 * cs[j].w;
          y[3] = a1 * cs[j].w + b1 * cs[j].z;
        }
        store_chunk(a.cache, a.cache_dtype, static_cast<size_t>(loc) * hd + c0, y);
      }
    }
  }
}

// One wave: as many blocks as can be resident at once (the warps then loop).
template <int kChunks>
int launch_resident(const NormRopeArgs& a, cudaStream_t stream) {
  // per device; a failed query is not cached (the fallback of one block per SM is used for this launch only)
  static std::atomic<int> cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return CKV_ERR_LAUNCH;
  const bool cached_dev = dev >= 0 && dev < 64;
  int per_sm = cached_dev ? cache[dev].load(std::memory_order_relaxed) : 0;
  if (per_sm == 0) {
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, norm_rope_store_kernel<kChunks>, kNrThreads, 0) ==
            cudaSuccess &&
        per_sm > 0) {
      if (cached_dev) cache[dev].store(per_sm, std::memory_order_relaxed);
    } else {
      cudaGetLastError();
      per_sm = 1;
    }
  }
  const uint32_t warps_per_cta = kNrThreads / 32;
  uint32_t grid = (a.capacity + warps_per_cta - 1) / warps_per_cta;
  grid = std::max<uint32_t>(1, std::min<uint32_t>(grid, static_cast<uint32_t>(per_sm * sm_count())));
  return launch_pdl(norm_rope_store_kernel<kChunks>, dim3(grid), dim3(kNrThreads), 0, stream, a);
}

int launch_norm_rope(const NormRopeArgs& a, cudaStream_t stream) {
  if (a.ratio != 4 && a.ratio != 128) return CKV_ERR_RATIO;
  if (a.head_dim <= 0 || a.head_dim % 128 != 0 || a.head_dim > 1024) return CKV_ERR_HEAD_DIM;
  // rope_dim: even, and a multiple of 4 so that a lane's 4-channel chunk is either all norm or all pairs
  if (a.rope_dim < 0 || a.rope_dim % 4 != 0 || a.rope_dim > a.head_dim) return CKV_ERR_HEAD_DIM;
  if ((a.in_dtype != CKV_F32 && a.in_dtype != CKV_BF16) || (a.cache_dtype != CKV_F32 && a.cache_dtype != CKV_BF16) ||
      (a.in_layout != CKV_OUT_TOKEN && a.in_layout != CKV_OUT_COMPACT))
    return CKV_ERR_DTYPE;
  if (!(a.eps > 0.0f) || !(a.eps < 1e30f)) return CKV_ERR_SIZE;
  if (a.capacity == 0) return CKV_OK;
  if (!aligned16(a.rows) || !aligned16(a.cache) || !aligned16(a.weight) || (a.rope_dim > 0 && !aligned16(a.freqs)) ||
      (reinterpret_cast<uintptr_t>(a.out_loc) & 7u) || a.out_loc == nullptr)
    return CKV_ERR_POINTER;
  if (a.decode ? !aligned16(a.plan_d) : !aligned16(a.plan_c)) return CKV_ERR_POINTER;
  if (a.d_counts && (reinterpret_cast<uintptr_t>(a.d_counts) & 3u)) return CKV_ERR_POINTER;
  switch (a.head_dim / 128) {
    case 1: return launch_resident<1>(a, stream);
    case 2: return launch_resident<2>(a, stream);
    case 3: return launch_resident<3>(a, stream);
    case 4: return launch_resident<4>(a, stream);
    case 5: return launch_resident<5>(a, stream);
    case 6: return launch_resident<6>(a, stream);
    case 7: return launch_resident<7>(a, stream);
    default: return launch_resident<8>(a, stream);
  }
}

}  // namespace
}  // namespace ckv

using namespace ckv;

extern "C" int ckv_norm_rope_store_prefill(int ratio, int head_dim, int rope_dim, int in_dtype, const void* rows,
                                           int in_layout, uint64_t n_rows, const ckv_compress_plan_t* plan_c,
                                           const uint32_t* d_counts, uint32_t capacity_c, const float* norm_weight,
                                           float eps, const float* freqs, uint32_t max_pos, const int64_t* out_loc,
                                           uint64_t n_out_loc, int cache_dtype, void* kv_cache, uint64_t cache_rows,
                                           uint32_t* d_status, ckv_stream_t stream) {
  NormRopeArgs a{};
  a.ratio = ratio;
  a.decode = 0;
  a.head_dim = head_dim;
  a.rope_dim = rope_dim;
  a.in_dtype = in_dtype;
  a.in_layout = in_layout;
  a.rows = rows;
  a.n_rows = n_rows;
  a.plan_c = plan_c;
  a.d_counts = d_counts;
  a.capacity = capacity_c;
  a.weight = norm_weight;
  a.eps = eps;
  a.freqs = freqs;
  a.max_pos = max_pos;
  a.out_loc = out_loc;
  a.n_loc = n_out_loc;
  a.cache_dtype = cache_dtype;
  a.cache = kv_cache;
  a.cache_rows = cache_rows;
  a.d_status = d_status;
  return launch_norm_rope(a, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" int ckv_norm_rope_store_decode(int ratio, int head_dim, int rope_dim, int in_dtype, const void* rows,
                                          const ckv_decode_plan_t* plan_d, uint32_t batch, const float* norm_weight,
                                          float eps, const float* freqs, uint32_t max_pos, const int64_t* out_loc,
                                          int cache_dtype, void* kv_cache, uint64_t cache_rows, uint32_t* d_status,
                                          ckv_stream_t stream) {
  NormRopeArgs a{};
  a.ratio = ratio;
  a.decode = 1;
  a.head_dim = head_dim;
  a.rope_dim = rope_dim;
  a.in_dtype = in_dtype;
  a.in_layout = CKV_OUT_COMPACT;
  a.rows = rows;
  a.n_rows = batch;
  a.plan_d = plan_d;
  a.capacity = batch;
  a.weight = norm_weight;
  a.eps = eps;
  a.freqs = freqs;
  a.max_pos = max_pos;
  a.out_loc = out_loc;
  a.n_loc = batch;
  a.cache_dtype = cache_dtype;
  a.cache = kv_cache;
  a.cache_rows = cache_rows;
  a.d_status = d_status;
  return launch_norm_rope(a, reinterpret_cast<cudaStream_t>(stream));
}
