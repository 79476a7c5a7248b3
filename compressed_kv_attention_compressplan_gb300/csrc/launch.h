// launch.h -- internal host-side launchers shared between the libckv
// translation units (not part of the public ABI).
#pragma once

#include <cuda.h>  // CUtensorMap (type only; the encoder is fetched from the driver at run time)
#include <cuda_runtime.h>
#include <stdint.h>

#include "ckv.h"  // include/ (on the include path)

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
  const ckv_decode_order_t* order;    // decode: boundary rows in row order (NULL: the kernel scans plan_d)
  const int64_t* rid_hint;            // the planner's rid / seq_lens (/ extend_lens: prefill), read before
  const int64_t* seq_hint;            //   the dependency wait to prefetch windows into L2 (NULL: no
  const int64_t* ext_hint;            //   prefetch)
  uint32_t hint_batch;                // prefill: entries of the hint arrays
  const uint32_t* d_counts;           // prefill
  uint32_t capacity;                  // prefill: capacity_c; decode: batch
  int out_layout;
  void* out;
  uint32_t* d_status;
  uint64_t wait_ns;  // limit of the kernels' ordinary waits on asynchronous copies
};

int sm_count();

// The limit, in ns, that launches made from now on give their kernels' ordinary
// waits on asynchronous copies (ckv_set_wait_limit_ns).
uint64_t wait_limit_ns();

// Encodes a tiled tensor map of `rank` dimensions (dims[0] innermost; strides
// in bytes for dims 1 .. rank-1; box extents per dimension) over `base`, of
// dtype CKV_F32 / CKV_BF16, no swizzle, no fill.  CKV_OK or CKV_ERR_LAUNCH.
int encode_tensor_map(CUtensorMap* map, int dtype, uint32_t rank, const void* base, const uint64_t* dims,
                      const uint64_t* strides_bytes, const uint32_t* box);

int launch_c4_pool_prefill(const PoolArgs& a, cudaStream_t s);
int launch_c4_decode(const PoolArgs& a, cudaStream_t s);

// The norm + RoPE + store half of the fused C4 decode (ckv_compress_decode_norm_rope_store).
struct DecodeNormArgs {
  int rope_dim;
  const float* weight;   // [head_dim]
  float eps;
  const float* freqs;    // [max_pos, rope_dim/2, 2]
  uint32_t max_pos;
  const int64_t* out_loc;  // [batch]
  int cache_dtype;
  void* cache;           // [cache_rows, head_dim]
  uint64_t cache_rows;
};

int launch_c4_decode_norm(const PoolArgs& a, const DecodeNormArgs& n, cudaStream_t s);
int launch_c128_pool_prefill(const PoolArgs& a, cudaStream_t s);
int launch_c128_decode(const PoolArgs& a, cudaStream_t s);

inline bool aligned16(const void* p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline int check_launch() { return cudaGetLastError() == cudaSuccess ? CKV_OK : CKV_ERR_LAUNCH; }

// Launches `kernel` on `s` with programmatic stream serialisation allowed: the
// grid may begin while the previous kernel on the stream finishes (the kernel
// itself waits, with griddepcontrol.wait, before it touches dependent data).
template <typename... KArgs, typename... Args>
int launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...) != cudaSuccess) {
    cudaGetLastError();
    return CKV_ERR_LAUNCH;
  }
  return check_launch();
}

}  // namespace ckv
