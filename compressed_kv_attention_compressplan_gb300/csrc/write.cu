// write.cu -- the prefill state write: state[write_loc] = input[ragged_id].
//
// c4.cuh c4_write / flash_c4_prefill<kWrite=true> and compressor_v2.py
// _c128_compress_prefill_write_kernel copy one whole kv_score row per write
// record.  Here one warp moves one row with 16-byte vector accesses; all of a
// lane's loads are issued before its stores.
#include <algorithm>

#include "common.cuh"
#include "launch.h"

namespace ckv {
namespace {

constexpr int kWriteThreads = 256;
constexpr int kWriteUnroll = 8;  // 8 x 16 B per lane per pass = 4 KB per warp pass

struct WriteArgs {
  uint8_t* state;
  uint64_t state_rows;
  const uint8_t* input;
  uint32_t num_q_tokens;
  const ckv_write_plan_t* plan_w;
  const uint32_t* d_counts;
  uint32_t cap_w;
  uint32_t row_bytes;  // multiple of 512 (head_dim % 128 == 0)
  uint32_t* d_status;
};

__global__ __launch_bounds__(kWriteThreads) void write_kernel(const WriteArgs a) {
  pdl_wait();  // the pool of this step must have finished reading the state
  pdl_release();
  const uint32_t lane = threadIdx.x & 31;
  const uint32_t warps_total = gridDim.x * (kWriteThreads / 32);
  const uint32_t n = count_or_capacity(a.d_counts, 1, a.cap_w);
  for (uint32_t k = blockIdx.x * (kWriteThreads / 32) + (threadIdx.x >> 5); k < n; k += warps_total) {
    const uint2 rec = __ldg(reinterpret_cast<const uint2*>(a.plan_w + k));
    const uint32_t ragged = rec.x;
    const int32_t loc = static_cast<int32_t>(rec.y);
    if (loc < 0 || ragged == kInvalidU32) continue;
    if (ragged >= a.num_q_tokens || static_cast<uint64_t>(loc) >= a.state_rows) {
      if (lane == 0) status_or(a.d_status, CKV_STATUS_BAD_INDEX);
      continue;
    }
    const uint8_t* src = a.input + static_cast<size_t>(ragged) * a.row_bytes;
    uint8_t* dst = a.state + static_cast<size_t>(loc) * a.row_bytes;
    for (uint32_t base = lane * 16; base < a.row_bytes; base += 32 * 16 * kWriteUnroll) {
      uint4 v[kWriteUnroll];
#pragma unroll
      for (int u = 0; u < kWriteUnroll; ++u) {
        const uint32_t off = base + u * 32 * 16;
        if (off < a.row_bytes) v[u] = ld_stream16(src + off);
      }
#pragma unroll
      for (int u = 0; u < kWriteUnroll; ++u) {
        const uint32_t off = base + u * 32 * 16;
        if (off < a.row_bytes) st16(dst + off, v[u]);
      }
    }
  }
}

}  // namespace
}  // namespace ckv

using namespace ckv;

extern "C" int ckv_compress_write(int ratio, int head_dim, int dtype, void* state, uint64_t state_rows,
                                  const void* kv_score_input, uint32_t num_q_tokens, const ckv_write_plan_t* plan_w,
                                  const uint32_t* d_counts, uint32_t capacity_w, uint32_t* d_status,
                                  ckv_stream_t stream) {
  if (ratio != 4 && ratio != 128) return CKV_ERR_RATIO;
  if (head_dim <= 0 || head_dim % 128 != 0 || head_dim > 1024) return CKV_ERR_HEAD_DIM;
  if (dtype != CKV_F32 && dtype != CKV_BF16) return CKV_ERR_DTYPE;
  if (capacity_w == 0) return CKV_OK;
  if (!aligned16(state) || !aligned16(kv_score_input) || plan_w == nullptr ||
      (reinterpret_cast<uintptr_t>(plan_w) & 7u) || (d_counts && (reinterpret_cast<uintptr_t>(d_counts) & 3u)))
    return CKV_ERR_POINTER;
  const uint32_t width = ratio == 4 ? 4 * head_dim : 2 * head_dim;
  WriteArgs a{static_cast<uint8_t*>(state), state_rows, static_cast<const uint8_t*>(kv_score_input), num_q_tokens,
              plan_w, d_counts, capacity_w, width * (dtype == CKV_BF16 ? 2u : 4u), d_status};
  const uint32_t warps_per_cta = kWriteThreads / 32;
  uint32_t grid = (capacity_w + warps_per_cta - 1) / warps_per_cta;
  grid = std::max<uint32_t>(1, std::min<uint32_t>(grid, 8u * static_cast<uint32_t>(sm_count())));
  return launch_pdl(write_kernel, dim3(grid), dim3(kWriteThreads), 0, reinterpret_cast<cudaStream_t>(stream), a);
}
