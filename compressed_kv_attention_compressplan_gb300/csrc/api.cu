// api.cu -- the compute entry points of the C ABI: argument checks on the
// host, then dispatch to the ratio-specific launchers.
#include <atomic>

#include "async_copy.cuh"
#include "common.cuh"
#include "launch.h"

using namespace ckv;

namespace {

std::atomic<uint64_t> g_wait_limit_ns{kWaitLimitNs};

int check_pool_args(int ratio, int head_dim, int in_dtype, int out_dtype) {
  if (ratio != 4 && ratio != 128) return CKV_ERR_RATIO;
  if (head_dim <= 0 || head_dim % 128 != 0 || head_dim > 1024) return CKV_ERR_HEAD_DIM;
  if ((in_dtype != CKV_F32 && in_dtype != CKV_BF16) || (out_dtype != CKV_F32 && out_dtype != CKV_BF16))
    return CKV_ERR_DTYPE;
  return CKV_OK;
}

}  // namespace

namespace ckv {

uint64_t wait_limit_ns() { return g_wait_limit_ns.load(std::memory_order_relaxed); }

}  // namespace ckv

extern "C" {

uint64_t ckv_set_wait_limit_ns(uint64_t limit_ns) {
  // a limit beyond the ceiling would make `now - start > limit` unreachable
  // in practice, i.e. the waits unbounded again
  const uint64_t v = limit_ns == 0 ? kWaitLimitNs : (limit_ns > kWaitLimitMaxNs ? kWaitLimitMaxNs : limit_ns);
  return g_wait_limit_ns.exchange(v, std::memory_order_relaxed);
}

int ckv_compress_pool_prefill(int ratio, int head_dim, int in_dtype, int out_dtype, const void* state,
                              uint64_t state_rows, const void* kv_score_input, uint32_t num_q_tokens,
                              const void* ape, const ckv_compress_plan_t* plan_c, const uint32_t* d_counts,
                              uint32_t capacity_c, int out_layout, void* out, const ckv_prefill_hints_t* hints,
                              uint32_t* d_status, ckv_stream_t stream) {
  int rc = check_pool_args(ratio, head_dim, in_dtype, out_dtype);
  if (rc) return rc;
  if (out_layout != CKV_OUT_TOKEN && out_layout != CKV_OUT_COMPACT) return CKV_ERR_DTYPE;
  if (num_q_tokens > CKV_MAX_TOKENS || capacity_c > CKV_MAX_TOKENS + 1u) return CKV_ERR_SIZE;
  const bool token = out_layout == CKV_OUT_TOKEN;
  if ((token ? num_q_tokens : capacity_c) == 0) return CKV_OK;
  if (!aligned16(out) || !aligned16(ape)) return CKV_ERR_POINTER;
  if (capacity_c > 0 && (!aligned16(plan_c) || !aligned16(kv_score_input) || !aligned16(state)))
    return CKV_ERR_POINTER;
  if (d_counts && (reinterpret_cast<uintptr_t>(d_counts) & 3u)) return CKV_ERR_POINTER;
  if (hints != nullptr && hints->batch > 0 &&
      (hints->rid == nullptr || hints->seq_lens == nullptr || hints->extend_lens == nullptr ||
       ((reinterpret_cast<uintptr_t>(hints->rid) | reinterpret_cast<uintptr_t>(hints->seq_lens) |
         reinterpret_cast<uintptr_t>(hints->extend_lens)) & 7u)))
    return CKV_ERR_POINTER;
  PoolArgs a{};
  a.ratio = ratio;
  a.head_dim = head_dim;
  a.in_dtype = in_dtype;
  a.out_dtype = out_dtype;
  a.state = state;
  a.state_rows = state_rows;
  a.input = kv_score_input;
  a.num_q_tokens = num_q_tokens;
  a.ape = ape;
  a.plan_c = plan_c;
  a.d_counts = d_counts;
  a.capacity = capacity_c;
  a.out_layout = out_layout;
  a.out = out;
  a.d_status = d_status;
  a.wait_ns = wait_limit_ns();
  if (hints != nullptr && hints->batch > 0 && capacity_c > 0 &&
      static_cast<uint64_t>(num_q_tokens) * (ratio == 4 ? 4u : 2u) * head_dim * (in_dtype == CKV_BF16 ? 2u : 4u) <=
          CKV_PREFILL_HINT_MAX_INPUT_BYTES) {
    a.rid_hint = hints->rid;
    a.seq_hint = hints->seq_lens;
    a.ext_hint = hints->extend_lens;
    a.hint_batch = hints->batch;
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  return ratio == 4 ? launch_c4_pool_prefill(a, s) : launch_c128_pool_prefill(a, s);
}

int ckv_compress_prefill(int ratio, int head_dim, int in_dtype, int out_dtype, void* state, uint64_t state_rows,
                         const void* kv_score_input, uint32_t num_q_tokens, const void* ape,
                         const ckv_compress_plan_t* plan_c, const ckv_write_plan_t* plan_w,
                         const uint32_t* d_counts, uint32_t capacity_c, uint32_t capacity_w, int out_layout,
                         void* out, const ckv_prefill_hints_t* hints, uint32_t* d_status, ckv_stream_t stream) {
  // validate both halves before launching either
  int rc = check_pool_args(ratio, head_dim, in_dtype, out_dtype);
  if (rc) return rc;
  if (capacity_w > 0 && (!aligned16(state) || !aligned16(kv_score_input) || plan_w == nullptr ||
                         (reinterpret_cast<uintptr_t>(plan_w) & 7u)))
    return CKV_ERR_POINTER;
  rc = ckv_compress_pool_prefill(ratio, head_dim, in_dtype, out_dtype, state, state_rows, kv_score_input,
                                 num_q_tokens, ape, plan_c, d_counts, capacity_c, out_layout, out, hints, d_status,
                                 stream);
  if (rc) return rc;
  return ckv_compress_write(ratio, head_dim, in_dtype, state, state_rows, kv_score_input, num_q_tokens, plan_w,
                            d_counts, capacity_w, d_status, stream);
}

int ckv_compress_decode(int ratio, int head_dim, int in_dtype, int out_dtype, void* state, uint64_t state_rows,
                        const void* kv_score_input, const void* ape, const ckv_decode_plan_t* plan_d,
                        const ckv_decode_order_t* order, const int64_t* rid_hint, const int64_t* seq_lens_hint,
                        uint32_t batch, void* out, uint32_t* d_status, ckv_stream_t stream) {
  int rc = check_pool_args(ratio, head_dim, in_dtype, out_dtype);
  if (rc) return rc;
  if (batch == 0) return CKV_OK;
  if (!aligned16(state) || !aligned16(kv_score_input) || !aligned16(ape) || !aligned16(plan_d) || !aligned16(out))
    return CKV_ERR_POINTER;
  if ((reinterpret_cast<uintptr_t>(order) | reinterpret_cast<uintptr_t>(rid_hint) |
       reinterpret_cast<uintptr_t>(seq_lens_hint)) & 7u)
    return CKV_ERR_POINTER;
  PoolArgs a{};
  a.ratio = ratio;
  a.head_dim = head_dim;
  a.in_dtype = in_dtype;
  a.out_dtype = out_dtype;
  a.state = state;
  a.state_mut = state;
  a.state_rows = state_rows;
  a.input = kv_score_input;
  a.num_q_tokens = batch;
  a.ape = ape;
  a.plan_d = plan_d;
  a.order = order;
  a.rid_hint = rid_hint != nullptr && seq_lens_hint != nullptr ? rid_hint : nullptr;
  a.seq_hint = rid_hint != nullptr && seq_lens_hint != nullptr ? seq_lens_hint : nullptr;
  a.capacity = batch;
  a.out_layout = CKV_OUT_TOKEN;
  a.out = out;
  a.d_status = d_status;
  a.wait_ns = wait_limit_ns();
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  return ratio == 4 ? launch_c4_decode(a, s) : launch_c128_decode(a, s);
}

int ckv_compress_decode_norm_rope_store(int ratio, int head_dim, int rope_dim, int in_dtype, void* state,
                                        uint64_t state_rows, const void* kv_score_input, const void* ape,
                                        const ckv_decode_plan_t* plan_d, const int64_t* rid_hint,
                                        const int64_t* seq_lens_hint, uint32_t batch, const float* norm_weight,
                                        float eps, const float* freqs, uint32_t max_pos, const int64_t* out_loc,
                                        int cache_dtype, void* kv_cache, uint64_t cache_rows, uint32_t* d_status,
                                        ckv_stream_t stream) {
  if (ratio != 4) return CKV_ERR_RATIO;
  int rc = check_pool_args(ratio, head_dim, in_dtype, CKV_F32);
  if (rc) return rc;
  if (rope_dim < 0 || rope_dim % 4 != 0 || rope_dim > head_dim) return CKV_ERR_HEAD_DIM;
  if (cache_dtype != CKV_F32 && cache_dtype != CKV_BF16) return CKV_ERR_DTYPE;
  if (!(eps > 0.0f) || !(eps < 1e30f)) return CKV_ERR_SIZE;
  if (batch == 0) return CKV_OK;
  if (!aligned16(state) || !aligned16(kv_score_input) || !aligned16(ape) || !aligned16(plan_d) ||
      !aligned16(norm_weight) || !aligned16(kv_cache) || (rope_dim > 0 && !aligned16(freqs)) || out_loc == nullptr)
    return CKV_ERR_POINTER;
  if ((reinterpret_cast<uintptr_t>(out_loc) | reinterpret_cast<uintptr_t>(rid_hint) |
       reinterpret_cast<uintptr_t>(seq_lens_hint)) & 7u)
    return CKV_ERR_POINTER;
  PoolArgs a{};
  a.ratio = ratio;
  a.head_dim = head_dim;
  a.in_dtype = in_dtype;
  a.out_dtype = CKV_F32;
  a.state = state;
  a.state_mut = state;
  a.state_rows = state_rows;
  a.input = kv_score_input;
  a.num_q_tokens = batch;
  a.ape = ape;
  a.plan_d = plan_d;
  a.rid_hint = rid_hint != nullptr && seq_lens_hint != nullptr ? rid_hint : nullptr;
  a.seq_hint = rid_hint != nullptr && seq_lens_hint != nullptr ? seq_lens_hint : nullptr;
  a.capacity = batch;
  a.out_layout = CKV_OUT_TOKEN;
  a.d_status = d_status;
  a.wait_ns = wait_limit_ns();
  DecodeNormArgs n{};
  n.rope_dim = rope_dim;
  n.weight = norm_weight;
  n.eps = eps;
  n.freqs = freqs;
  n.max_pos = max_pos;
  n.out_loc = out_loc;
  n.cache_dtype = cache_dtype;
  n.cache = kv_cache;
  n.cache_rows = cache_rows;
  return launch_c4_decode_norm(a, n, reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"
