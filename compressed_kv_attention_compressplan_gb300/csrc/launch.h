// launch.h -- internal host-side launchers shared between the libckv
// translation units (not part of the public ABI).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/ckv.h"

namespace ckv {

// Arguments of the pooling kernels (prefill and decode, both ratios).
struct PoolArgs {
  int ratio;
  int head_dim;
  int in_dtype;
  int out_dtype;
  const void* state;        // pool prefill: read only
  void* state_mut;          // decode: written (the new token's row)
  uint64_t state_rows;
  const void* input;
  uint32_t num_q_tokens;    // prefill: rows of input; decode: batch
  const void* ape;
  const ckv_compress_plan_t* plan_c;  // prefill
  const ckv_decode_plan_t* plan_d;    // decode
  const uint32_t* d_counts;           // prefill
  uint32_t capacity;                  // prefill: capacity_c; decode: batch
  int out_layout;
  void* out;
  uint32_t* d_status;
};

int sm_count();

int launch_c4_pool_prefill(const PoolArgs& a, cudaStream_t s);
int launch_c4_decode(const PoolArgs& a, cudaStream_t s);
int launch_c128_pool_prefill(const PoolArgs& a, cudaStream_t s);
int launch_c128_decode(const PoolArgs& a, cudaStream_t s);

inline bool aligned16(const void* p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline int check_launch() { return cudaGetLastError() == cudaSuccess ? CKV_OK : CKV_ERR_LAUNCH; }

}  // namespace ckv
