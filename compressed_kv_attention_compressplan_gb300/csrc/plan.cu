// plan.cu -- the plan builders (decode and prefill) and small host helpers.
//
// Prefill planning follows the sequential CPU loop of c_plan.cuh
// plan_compress_prefill_legacy (requests in batch order, positions ascending,
// compress and write records in separate lists) together with the legacy
// ring / page translation of plan_compress_prefill_legacy_kernel, or, for
// SWA-paged state, the loop and translation of plan_compress_prefill /
// plan_compress_prefill_kernel_1.  c_plan.cuh's own GPU builder
// (plan_compress_prefill_kernel0) walks requests serially inside
// one CTA and hands out slots with shared-memory atomics, so its order varies
// run to run.  Here every record's index is a closed form of block-wide
// exclusive scans of the per-request counts, so the GPU plan is bit-identical
// to the CPU loop, and the work is O(records) spread over the whole grid.
#include <algorithm>
#include <atomic>

#include "common.cuh"
#include "launch.h"

namespace ckv {

namespace {

constexpr int kPlanThreads = 1024;  // one thread per request (batch <= 1024)
constexpr int kWarps = kPlanThreads / 32;

__device__ __forceinline__ int32_t legacy_page(int ratio, int32_t rid, int32_t position) {
  // c_plan.cuh legacy_compute_page: C4 uses two 4-slot pages per request,
  // alternating with the group index; C128 uses one page per request.
  return ratio == 4 ? rid * 2 + ((position / 4) & 1) : rid;
}

__device__ __forceinline__ int32_t legacy_loc(int ratio, int32_t rid, int32_t position) {
  return legacy_page(ratio, rid, position) * ratio + position % ratio;
}

// Inclusive warp scan of a 32-bit value (Kogge-Stone over __shfl_up_sync).
__device__ __forceinline__ uint32_t warp_inclusive_sum(uint32_t v, int lane) {
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const uint32_t n = __shfl_up_sync(0xFFFFFFFFu, v, off);
    if (lane >= off) v += n;
  }
  return v;
}

__device__ __forceinline__ unsigned long long warp_inclusive_sum64(unsigned long long v, int lane) {
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const unsigned long long n = __shfl_up_sync(0xFFFFFFFFu, v, off);
    if (lane >= off) v += n;
  }
  return v;
}

__device__ __forceinline__ uint32_t warp_max(uint32_t v) {
#pragma unroll
  for (int m = 16; m > 0; m >>= 1) v = max(v, __shfl_xor_sync(0xFFFFFFFFu, v, m));
  return v;
}

__device__ __forceinline__ uint32_t warp_min(uint32_t v) {
#pragma unroll
  for (int m = 16; m > 0; m >>= 1) v = min(v, __shfl_xor_sync(0xFFFFFFFFu, v, m));
  return v;
}

// The legacy DecodePlan record of one row (c_plan.cuh
// plan_compress_decode_legacy_kernel); rows with bad lengths get the invalid
// record and set CKV_STATUS_BAD_LENGTH.
__device__ __forceinline__ uint4 legacy_decode_record(int ratio, int64_t sl, int64_t r, uint32_t* d_status) {
  const int64_t slots = ratio == 4 ? 8 : 128;
  if (sl >= 1 && sl <= INT32_MAX && r >= 0 && r * slots + slots - 1 <= INT32_MAX) {
    const int32_t p1 = static_cast<int32_t>(sl - 1);
    const int32_t p0 = max(p1 - ratio, 0);
    const int32_t rr = static_cast<int32_t>(r);
    return make_uint4(static_cast<uint32_t>(sl), static_cast<uint32_t>(legacy_loc(ratio, rr, p1)),
                      static_cast<uint32_t>(legacy_page(ratio, rr, p0)),
                      static_cast<uint32_t>(legacy_page(ratio, rr, p1)));
  }
  status_or(d_status, CKV_STATUS_BAD_LENGTH);
  return make_uint4(kInvalidU32, kInvalidU32, kInvalidU32, kInvalidU32);
}

__global__ void plan_decode_kernel(int ratio, const int64_t* __restrict__ rid, const int64_t* __restrict__ seq_lens,
                                   uint32_t batch, ckv_decode_plan_t* __restrict__ plan_d, uint32_t* d_status) {
  pdl_release();  // the decode may launch at once and warm the L2 (see plan_decode_ordered_kernel)
  pdl_wait();
  const uint32_t b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= batch) return;
  *reinterpret_cast<uint4*>(plan_d + b) = legacy_decode_record(ratio, seq_lens[b], rid[b], d_status);
}

// The boundary list of a decode batch next to its records: one CTA of
// kPlanThreads threads walks the batch in chunks of K * kPlanThreads rows
// (thread t takes rows chunk + K*t .. chunk + K*t + K-1), and a block-wide
// exclusive scan of the per-thread counts of valid records with
// seq_len % ratio == 0 places each such row's entry {row, read_page_0}, so
// the list is in row order.  order[0] = {count, 0}.  rec_of(b) computes row
// b's record (its loads are issued for all K rows before any is used).
template <int K, typename RecOf>
__device__ __forceinline__ void plan_decode_ordered_body(int ratio, uint32_t batch, ckv_decode_plan_t* plan_d,
                                                         ckv_decode_order_t* order, RecOf rec_of) {
  __shared__ uint32_t s_warp[kWarps];
  const int t = threadIdx.x;
  const int lane = t & 31;
  const int warp = t >> 5;
  uint32_t base = 0;
  for (uint32_t chunk = 0; chunk < batch; chunk += K * kPlanThreads) {
    uint4 rec[K];
    bool take[K];
    uint32_t cnt = 0;
    rec_of(chunk + K * t, rec);
#pragma unroll
    for (int k = 0; k < K; ++k) {
      const uint32_t b = chunk + K * t + k;
      take[k] = false;
      if (b < batch) {
        *reinterpret_cast<uint4*>(plan_d + b) = rec[k];
        take[k] = rec[k].x != kInvalidU32 && rec[k].x % static_cast<uint32_t>(ratio) == 0;
      }
      cnt += take[k] ? 1u : 0u;
    }
    const uint32_t incl = warp_inclusive_sum(cnt, lane);
    if (lane == 31) s_warp[warp] = incl;
    __syncthreads();
    uint32_t pos = base + incl - cnt, total = 0;
#pragma unroll 8
    for (int w = 0; w < kWarps; ++w) {
      const uint32_t v = s_warp[w];
      if (w < warp) pos += v;
      total += v;
    }
#pragma unroll
    for (int k = 0; k < K; ++k) {
      if (take[k]) {
        *reinterpret_cast<uint2*>(order + 1 + pos) = make_uint2(chunk + K * t + k, rec[k].z);
        ++pos;
      }
    }
    base += total;
    __syncthreads();  // s_warp is rewritten by the next chunk
  }
  if (t == 0) *reinterpret_cast<uint2*>(order) = make_uint2(base, 0u);
}

template <int K>
__global__ __launch_bounds__(kPlanThreads, 1) void plan_decode_ordered_kernel(
    int ratio, const int64_t* __restrict__ rid, const int64_t* __restrict__ seq_lens, uint32_t batch,
    ckv_decode_plan_t* __restrict__ plan_d, ckv_decode_order_t* __restrict__ order, uint32_t* d_status) {
  // the decode that follows may launch at once: its CTAs then warm the L2
  // while this kernel and its predecessor finish
  pdl_release();
  pdl_wait();
  plan_decode_ordered_body<K>(ratio, batch, plan_d, order, [&](uint32_t b0, uint4 (&rec)[K]) {
    int64_t sl[K], r[K];
#pragma unroll
    for (int k = 0; k < K; ++k) {
      sl[k] = b0 + k < batch ? seq_lens[b0 + k] : 0;
      r[k] = b0 + k < batch ? rid[b0 + k] : 0;
    }
#pragma unroll
    for (int k = 0; k < K; ++k)
      rec[k] = b0 + k < batch ? legacy_decode_record(ratio, sl[k], r[k], d_status) : make_uint4(0, 0, 0, 0);
  });
}

// c_plan.cuh compute_loc: an SWA slot swa lives in the ring of its SWA page,
// state row = (swa / swa_page_size) * ring_size + swa % ring_size.
__device__ __forceinline__ int64_t paged_loc(const int32_t* r2t, int64_t stride, const int64_t* f2s,
                                             uint64_t num_full, int32_t sps, int32_t ring, int32_t rid, int32_t p,
                                             bool& ok) {
  const int32_t raw = r2t[static_cast<int64_t>(rid) * stride + p];
  if (raw < 0 || static_cast<uint64_t>(raw) >= num_full) {
    ok = false;
    return -1;
  }
  const int64_t swa = f2s[raw];
  const int64_t loc = swa >= 0 ? (swa / sps) * ring + swa % ring : -1;
  if (loc < 0 || loc > INT32_MAX - 4) {
    ok = false;
    return -1;
  }
  return loc;
}

// Positions x' < x with x' % S >= S - 4: the last group of every SWA page,
// which paged C4 always writes (c_plan.cuh plan_compress_prefill, should_write).
__device__ __forceinline__ int32_t page_end_count(int32_t x, int32_t S) {
  return (x / S) * 4 + max(0, x % S - (S - 4));
}

struct DecodePagedArgs {
  const int64_t* rid;
  const int64_t* seq_lens;
  uint32_t batch;
  const int32_t* r2t;
  int64_t r2t_stride;
  uint32_t num_reqs;
  const int64_t* f2s;
  uint64_t num_full;
  int32_t sps;
  int32_t ring;
  ckv_decode_plan_t* plan_d;
  uint32_t* d_status;
};

// c_plan.cuh plan_compress_decode_kernel (C4 through the SWA mapping):
// write_loc = ring(state of position seq_len-1), read pages of positions
// max(seq_len-1-4, 0) and seq_len-1.
__device__ __forceinline__ uint4 paged_decode_record(const DecodePagedArgs& a, int64_t sl, int64_t r) {
  uint4 rec = make_uint4(kInvalidU32, kInvalidU32, kInvalidU32, kInvalidU32);
  if (sl >= 1 && sl <= INT32_MAX && r >= 0) {
    if (r < a.num_reqs && sl <= a.r2t_stride) {
      const int32_t p1 = static_cast<int32_t>(sl - 1);
      const int32_t p0 = max(p1 - 4, 0);
      bool ok = true;
      const int64_t loc1 = paged_loc(a.r2t, a.r2t_stride, a.f2s, a.num_full, a.sps, a.ring, static_cast<int32_t>(r), p1, ok);
      const int64_t loc0 = paged_loc(a.r2t, a.r2t_stride, a.f2s, a.num_full, a.sps, a.ring, static_cast<int32_t>(r), p0, ok);
      if (ok)
        rec = make_uint4(static_cast<uint32_t>(sl), static_cast<uint32_t>(loc1), static_cast<uint32_t>(loc0 / 4),
                         static_cast<uint32_t>(loc1 / 4));
      else
        status_or(a.d_status, CKV_STATUS_BAD_INDEX);
    } else {
      status_or(a.d_status, CKV_STATUS_BAD_INDEX);
    }
  } else {
    status_or(a.d_status, CKV_STATUS_BAD_LENGTH);
  }
  return rec;
}

__global__ void plan_decode_paged_kernel(const DecodePagedArgs a) {
  pdl_wait();
  pdl_release();
  const uint32_t b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= a.batch) return;
  *reinterpret_cast<uint4*>(a.plan_d + b) = paged_decode_record(a, a.seq_lens[b], a.rid[b]);
}

template <int K>
__global__ __launch_bounds__(kPlanThreads, 1) void plan_decode_paged_ordered_kernel(const DecodePagedArgs a,
                                                                                   ckv_decode_order_t* order) {
  pdl_release();  // as plan_decode_ordered_kernel
  pdl_wait();
  plan_decode_ordered_body<K>(4, a.batch, a.plan_d, order, [&](uint32_t b0, uint4 (&rec)[K]) {
    int64_t sl[K], r[K];
#pragma unroll
    for (int k = 0; k < K; ++k) {
      sl[k] = b0 + k < a.batch ? a.seq_lens[b0 + k] : 0;
      r[k] = b0 + k < a.batch ? a.rid[b0 + k] : 0;
    }
#pragma unroll
    for (int k = 0; k < K; ++k) rec[k] = b0 + k < a.batch ? paged_decode_record(a, sl[k], r[k]) : make_uint4(0, 0, 0, 0);
  });
}

struct PrefillPlanArgs {
  int ratio;
  const int64_t* rid;
  const int64_t* seq_lens;
  const int64_t* extend_lens;
  uint32_t batch;
  uint32_t num_q_tokens;
  uint32_t cap_c;
  uint32_t cap_w;
  int pad_invalid;
  ckv_compress_plan_t* plan_c;
  ckv_write_plan_t* plan_w;
  uint32_t* d_counts;
  uint32_t* d_status;
  // SWA-paged C4 addressing (paged != 0): state row of position p of request
  // rid = ring(full_to_state[req_to_token[rid][p]]), see paged_loc.
  int paged;
  const int32_t* r2t;
  int64_t r2t_stride;
  uint32_t num_reqs;
  const int64_t* f2s;
  uint64_t num_full;
  int32_t sps;
  int32_t ring;
  // Online C128 state (online != 0): the second list holds one unit record per
  // (request, 128-group touched by the extend) instead of write records.
  int online;
  int64_t slot_offset;
  ckv_online_unit_t* units;
};

// Every CTA loads the <= 1024 request lengths, derives per request
//   pl = sl - el, nc = sl/R - pl/R, first_w = (sl/R)*R - (R == 4 ? 4 : 0),
//   wstart = max(pl, first_w), nw = sl - wstart,
// scans el, nc and nw (exclusive, block-wide), reduces min / max of el, and
// then emits records k = global thread, global thread + grid stride, ...:
// record k of the compress list belongs to the request b with
// off_c[b] <= k < off_c[b+1] (binary search), whose (k - off_c[b])-th event is
// at position (pl/R + k - off_c[b] + 1) * R - 1.  Likewise for writes, which
// cover positions wstart .. sl-1.  Built per ratio, so that every division by
// R is a shift (the kernel is a chain of dependent steps, 32 warps per CTA).
template <int kR>
__global__ __launch_bounds__(kPlanThreads, 1) void plan_prefill_kernel(const PrefillPlanArgs a) {
  __shared__ uint32_t s_off_c[kMaxBatch + 1];
  __shared__ uint32_t s_off_w[kMaxBatch + 1];
  __shared__ uint32_t s_off_e[kMaxBatch + 1];
  __shared__ int32_t s_pl[kMaxBatch];
  __shared__ int32_t s_wstart[kMaxBatch];
  __shared__ int32_t s_rid[kMaxBatch];
  __shared__ int32_t s_pe0[kMaxBatch];      // paged: page_end_count(prefix)
  __shared__ uint32_t s_nextra[kMaxBatch];  // paged: page-end writes before wstart
  __shared__ uint32_t s_wsum[3][kWarps];
  __shared__ uint32_t s_wmin[kWarps], s_wmax[kWarps];
  __shared__ uint32_t s_flags;
  __shared__ unsigned long long s_total_e;

  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  constexpr int R = kR;
  constexpr int64_t slots = R == 4 ? 8 : 128;
  if (tid == 0) s_flags = 0;
  pdl_wait();
  pdl_release();

  uint32_t el_eff = 0, nc = 0, nw = 0;
  uint32_t el_min = kInvalidU32, el_max = 0;
  if (tid < static_cast<int>(a.batch)) {
    const int64_t sl = a.seq_lens[tid];
    const int64_t el = a.extend_lens[tid];
    const int64_t r = a.rid[tid];
    const bool ok = el > 0 && el <= sl && sl <= INT32_MAX && r >= 0 && el <= CKV_MAX_TOKENS &&
                    (a.online ? r + a.slot_offset >= 0 && r + a.slot_offset <= INT32_MAX
                              : r * slots + slots - 1 <= INT32_MAX);
    el_eff = (el > 0 && el <= CKV_MAX_TOKENS) ? static_cast<uint32_t>(el) : 0u;
    el_min = el_max = el_eff;
    bool ok_paged = true;
    if (ok && a.paged && R == 4) ok_paged = r < a.num_reqs && sl <= a.r2t_stride;
    if (ok && ok_paged) {
      const int32_t s32 = static_cast<int32_t>(sl);
      const int32_t pl = s32 - static_cast<int32_t>(el);
      int32_t first_w = (s32 / R) * R - (R == 4 ? 4 : 0);
      uint32_t nextra = 0;
      int32_t pe0 = 0;
      if (a.paged) {
        // c_plan.cuh's GPU-input planner also keeps the last mtp_pad positions
        const int32_t mtp_pad = min(a.ring - R, 4);
        first_w = min(first_w, s32 - mtp_pad);
      }
      const int32_t wstart = max(pl, first_w);
      if (a.paged && R == 4 && wstart > pl) {
        pe0 = page_end_count(pl, a.sps);
        nextra = static_cast<uint32_t>(page_end_count(wstart, a.sps) - pe0);
      }
      nc = static_cast<uint32_t>(s32 / R - pl / R);
      nw = static_cast<uint32_t>(s32 - wstart) + nextra;
      if (a.online) {  // units: the 128-groups pl/128 .. (sl-1)/128; wstart keeps sl
        nw = static_cast<uint32_t>((s32 - 1) / 128 - pl / 128 + 1);
        s_wstart[tid] = s32;
      }
      s_pl[tid] = pl;
      if (!a.online) s_wstart[tid] = wstart;
      s_rid[tid] = static_cast<int32_t>(r);
      s_pe0[tid] = pe0;
      s_nextra[tid] = nextra;
    } else {
      s_pl[tid] = 0;
      s_wstart[tid] = 0;
      s_rid[tid] = 0;
      s_pe0[tid] = 0;
      s_nextra[tid] = 0;
      if (ok) atomicOr(&s_flags, CKV_STATUS_BAD_INDEX);
    }
    if (!ok) atomicOr(&s_flags, CKV_STATUS_BAD_LENGTH);
  }

  // Block-wide exclusive scans of (el_eff, nc, nw): warp scans, then a scan of
  // the 32 warp totals by warp 0.  A warp's token sum is below 32 * 2^24; the
  // token grand total is also formed in 64 bits so that garbage lengths cannot
  // wrap around to a plausible total (records are only emitted when it equals
  // num_q_tokens < 2^24, and then no partial sum can overflow).  (Every thread
  // adding up the warp totals itself instead, one barrier less, was slower:
  // 5.3 against 3.0 us back to back.)
  const uint32_t ie = warp_inclusive_sum(el_eff, lane);
  const uint32_t ic = warp_inclusive_sum(nc, lane);
  const uint32_t iw = warp_inclusive_sum(nw, lane);
  const uint32_t wmn = warp_min(el_min), wmx = warp_max(el_max);
  if (lane == 31) {
    s_wsum[0][warp] = ie;
    s_wsum[1][warp] = ic;
    s_wsum[2][warp] = iw;
  }
  if (lane == 0) {
    s_wmin[warp] = wmn;
    s_wmax[warp] = wmx;
  }
  __syncthreads();
  if (warp == 0) {
    const uint32_t te = warp_inclusive_sum(s_wsum[0][lane], lane);
    const unsigned long long te64 = warp_inclusive_sum64(s_wsum[0][lane], lane);
    const uint32_t tc = warp_inclusive_sum(s_wsum[1][lane], lane);
    const uint32_t tw = warp_inclusive_sum(s_wsum[2][lane], lane);
    const uint32_t mn = warp_min(s_wmin[lane]), mx = warp_max(s_wmax[lane]);
    s_wsum[0][lane] = te - s_wsum[0][lane];  // exclusive warp offsets
    s_wsum[1][lane] = tc - s_wsum[1][lane];
    s_wsum[2][lane] = tw - s_wsum[2][lane];
    if (lane == 31) {
      s_total_e = te64;
      s_off_e[kMaxBatch] = te;
      s_off_c[kMaxBatch] = tc;
      s_off_w[kMaxBatch] = tw;
    }
    if (lane == 0) {
      s_wmin[0] = mn;
      s_wmax[0] = mx;
    }
  }
  __syncthreads();
  s_off_e[tid] = s_wsum[0][warp] + ie - el_eff;
  s_off_c[tid] = s_wsum[1][warp] + ic - nc;
  s_off_w[tid] = s_wsum[2][warp] + iw - nw;
  __syncthreads();

  const uint32_t B = a.batch;
  const unsigned long long total_e = s_total_e;
  const uint32_t num_c = s_off_c[kMaxBatch];
  const uint32_t num_w = s_off_w[kMaxBatch];
  const uint32_t e_min = s_wmin[0], e_max = s_wmax[0];
  if (blockIdx.x == 0 && tid == 0) {
    uint32_t flags = s_flags;
    if (total_e != a.num_q_tokens) flags |= CKV_STATUS_BAD_TOTAL;
    if ((!a.online && num_c > a.cap_c) || num_w > a.cap_w) flags |= CKV_STATUS_CAPACITY;
    if (flags) status_or(a.d_status, flags);
    a.d_counts[0] = num_c;
    a.d_counts[1] = num_w;
    a.d_counts[2] = B ? e_min : 0u;
    a.d_counts[3] = B ? e_max : 0u;
  }
  // Entries past the end of a short ragged buffer would name rows that do not
  // exist: with a bad token total, emit nothing but padding.
  const bool usable = total_e == a.num_q_tokens;
  const uint32_t emit_c = usable ? min(num_c, a.cap_c) : 0u;
  const uint32_t emit_w = usable ? min(num_w, a.cap_w) : 0u;
  constexpr int W = R == 4 ? 8 : 128;

  const uint32_t stride = gridDim.x * blockDim.x;
  const uint32_t work = max(a.cap_c, a.cap_w);
  // The pages' MTP-uniform case on the legacy layout (every extend_len equal
  // to some e <= 32: the speculative-decoding verify step): token t is position
  // t % e of request t / e, so the records are emitted per token in closed
  // form -- a compress record where (p + 1) % R == 0, at the request's offset
  // plus the events before it; a write record where p >= wstart, at the
  // request's offset plus p - wstart -- with no search, and the padding
  // follows in a grid-stride loop.  The records and their places are those of
  // the search below.
  if (!a.paged && !a.online && B > 0 && e_min == e_max && e_max > 0 && e_max <= 32 && usable) {
    const uint32_t e = e_max;
    const uint32_t tokens = B * e;  // == num_q_tokens (usable)
    for (uint32_t t = blockIdx.x * blockDim.x + tid; t < tokens; t += stride) {
      const uint32_t b = t / e;
      const int32_t pl = s_pl[b];
      const int32_t j = static_cast<int32_t>(t - b * e);
      const int32_t p = pl + j;
      const int32_t rid = s_rid[b];
      if ((p + 1) % R == 0) {
        const uint32_t k = s_off_c[b] + static_cast<uint32_t>((p + 1) / R - pl / R - 1);
        if (k < emit_c && k < s_off_c[b + 1]) {
          const uint32_t bl = static_cast<uint32_t>(W - min(j + 1, W));
          *reinterpret_cast<uint4*>(a.plan_c + k) =
              make_uint4(static_cast<uint32_t>(p + 1), t | (bl << CKV_BUFFER_LEN_SHIFT),
                         static_cast<uint32_t>(legacy_page(R, rid, max(p - R, 0))),
                         static_cast<uint32_t>(legacy_page(R, rid, p)));
        }
      }
      const int32_t ws = s_wstart[b];
      if (p >= ws) {
        const uint32_t k = s_off_w[b] + static_cast<uint32_t>(p - ws);
        if (k < emit_w && k < s_off_w[b + 1])
          *reinterpret_cast<uint2*>(a.plan_w + k) = make_uint2(t, static_cast<uint32_t>(legacy_loc(R, rid, p)));
      }
    }
    if (a.pad_invalid) {
      for (uint32_t k = blockIdx.x * blockDim.x + tid; k < work; k += stride) {
        if (k >= emit_c && k < a.cap_c)
          *reinterpret_cast<uint4*>(a.plan_c + k) = make_uint4(kInvalidU32, kInvalidU32, kInvalidU32, kInvalidU32);
        if (k >= emit_w && k < a.cap_w) *reinterpret_cast<uint2*>(a.plan_w + k) = make_uint2(kInvalidU32, kInvalidU32);
      }
    }
    return;
  }
  for (uint32_t k = blockIdx.x * blockDim.x + tid; k < work; k += stride) {
    if (k < a.cap_c) {
      uint4 rec = make_uint4(kInvalidU32, kInvalidU32, kInvalidU32, kInvalidU32);
      bool store = a.pad_invalid != 0;
      if (k < emit_c) {
        uint32_t lo = 0, hi = B;  // largest b with off_c[b] <= k
        while (hi - lo > 1) {
          const uint32_t mid = (lo + hi) >> 1;
          if (s_off_c[mid] <= k) lo = mid; else hi = mid;
        }
        const int32_t pl = s_pl[lo];
        const int32_t p = (pl / R + static_cast<int32_t>(k - s_off_c[lo]) + 1) * R - 1;
        const int32_t j = p - pl;
        const uint32_t ragged = s_off_e[lo] + static_cast<uint32_t>(j);
        const uint32_t bl = static_cast<uint32_t>(W - min(j + 1, W));
        const int32_t rid = s_rid[lo];
        int64_t page0, page1;
        bool ok = true;
        if (a.paged && bl == 0) {  // reads no state; c_plan.cuh kernel_1 leaves (-1, batch index)
          page0 = -1;
          page1 = static_cast<int64_t>(lo);
        } else if (a.paged && R == 4) {
          page0 = paged_loc(a.r2t, a.r2t_stride, a.f2s, a.num_full, a.sps, a.ring, rid, max(p - R, 0), ok) / R;
          page1 = paged_loc(a.r2t, a.r2t_stride, a.f2s, a.num_full, a.sps, a.ring, rid, p, ok) / R;
        } else {
          page0 = legacy_page(R, rid, max(p - R, 0));
          page1 = legacy_page(R, rid, p);
        }
        if (ok) {
          rec = make_uint4(static_cast<uint32_t>(p + 1), ragged | (bl << CKV_BUFFER_LEN_SHIFT),
                           static_cast<uint32_t>(page0), static_cast<uint32_t>(page1));
        } else {
          status_or(a.d_status, CKV_STATUS_BAD_INDEX);
        }
        store = true;
      }
      if (store) *reinterpret_cast<uint4*>(a.plan_c + k) = rec;
    }
    if (a.online && k < a.cap_w) {
      uint4 rec = make_uint4(kInvalidU32, kInvalidU32, kInvalidU32, kInvalidU32);
      bool store = a.pad_invalid != 0;
      if (k < emit_w) {
        uint32_t lo = 0, hi = B;
        while (hi - lo > 1) {
          const uint32_t mid = (lo + hi) >> 1;
          if (s_off_w[mid] <= k) lo = mid; else hi = mid;
        }
        const uint32_t kk = k - s_off_w[lo];
        const int32_t pl = s_pl[lo], sl = s_wstart[lo];
        const int32_t g = pl / 128 + static_cast<int32_t>(kk);
        const int32_t p0 = max(pl, 128 * g), p1 = min(sl, 128 * g + 128);
        const bool emit = p1 == 128 * g + 128;
        const uint32_t flags = (p0 % 128 != 0 ? CKV_UNIT_LOAD : 0u) | (emit ? CKV_UNIT_EMIT : 0u) |
                               (p1 == sl ? CKV_UNIT_STORE : 0u);
        rec = make_uint4(static_cast<uint32_t>(p0),
                         (s_off_e[lo] + static_cast<uint32_t>(p0 - pl)) |
                             (static_cast<uint32_t>(p1 - p0) << CKV_UNIT_COUNT_SHIFT),
                         static_cast<uint32_t>(s_rid[lo] + a.slot_offset),
                         (emit ? s_off_c[lo] + kk : CKV_RAGGED_MASK) | (flags << CKV_UNIT_FLAGS_SHIFT));
        store = true;
      }
      if (store) *reinterpret_cast<uint4*>(a.units + k) = rec;
    } else if (k < a.cap_w) {
      uint2 rec = make_uint2(kInvalidU32, kInvalidU32);
      bool store = a.pad_invalid != 0;
      if (k < emit_w) {
        uint32_t lo = 0, hi = B;
        while (hi - lo > 1) {
          const uint32_t mid = (lo + hi) >> 1;
          if (s_off_w[mid] <= k) lo = mid; else hi = mid;
        }
        const uint32_t kk = k - s_off_w[lo];
        const uint32_t nx = s_nextra[lo];
        int32_t p;
        if (kk < nx) {  // the kk-th last-group position of an SWA page before wstart
          const int32_t m = s_pe0[lo] + static_cast<int32_t>(kk);
          p = (m / 4) * a.sps + (a.sps - 4) + m % 4;
        } else {
          p = s_wstart[lo] + static_cast<int32_t>(kk - nx);
        }
        const uint32_t ragged = s_off_e[lo] + static_cast<uint32_t>(p - s_pl[lo]);
        bool ok = true;
        const int64_t loc = a.paged && R == 4 ? paged_loc(a.r2t, a.r2t_stride, a.f2s, a.num_full, a.sps, a.ring, s_rid[lo], p, ok)
                                    : legacy_loc(R, s_rid[lo], p);
        if (ok) rec = make_uint2(ragged, static_cast<uint32_t>(loc));
        else status_or(a.d_status, CKV_STATUS_BAD_INDEX);
        store = true;
      }
      if (store) *reinterpret_cast<uint2*>(a.plan_w + k) = rec;
    }
  }
}

}  // namespace

int sm_count() {
  static std::atomic<int> cached[64];  // per device (racing first calls store the same value)
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (dev < 0 || dev >= 64) return 148;
  int n = cached[dev].load(std::memory_order_relaxed);
  if (n == 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
      cudaGetLastError();
      return 148;  // not cached: a later call asks again
    }
    cached[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

}  // namespace ckv

using namespace ckv;

extern "C" {

uint32_t ckv_capacity_compress(int ratio, uint32_t batch, uint32_t num_q_tokens) {
  if (ratio != 4 && ratio != 128) return 0;
  const uint64_t c = static_cast<uint64_t>(num_q_tokens) / ratio + batch;
  return static_cast<uint32_t>(std::min<uint64_t>(c, num_q_tokens));
}

uint32_t ckv_capacity_write(int ratio, uint32_t batch, uint32_t num_q_tokens) {
  if (ratio != 4 && ratio != 128) return 0;
  const uint64_t w = static_cast<uint64_t>(batch) * (ratio == 4 ? 7 : 127);
  return static_cast<uint32_t>(std::min<uint64_t>(w, num_q_tokens));
}

int ckv_plan_decode(int ratio, const int64_t* rid, const int64_t* seq_lens, uint32_t batch,
                    ckv_decode_plan_t* plan_d, ckv_decode_order_t* order, uint32_t* d_status, ckv_stream_t stream) {
  if (ratio != 4 && ratio != 128) return CKV_ERR_RATIO;
  if (batch == 0 && order == nullptr) return CKV_OK;
  if (batch > 0 && (!rid || !seq_lens || !aligned16(plan_d))) return CKV_ERR_POINTER;
  if ((reinterpret_cast<uintptr_t>(rid) | reinterpret_cast<uintptr_t>(seq_lens)) & 7u) return CKV_ERR_POINTER;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (order != nullptr) {
    if (reinterpret_cast<uintptr_t>(order) & 7u) return CKV_ERR_POINTER;
    // one CTA: the list is a block-wide scan over the whole batch
    if (batch <= kPlanThreads)
      return launch_pdl(plan_decode_ordered_kernel<1>, dim3(1), dim3(kPlanThreads), 0, s, ratio, rid, seq_lens, batch,
                        plan_d, order, d_status);
    return launch_pdl(plan_decode_ordered_kernel<4>, dim3(1), dim3(kPlanThreads), 0, s, ratio, rid, seq_lens, batch,
                      plan_d, order, d_status);
  }
  const uint32_t threads = 256;
  return launch_pdl(plan_decode_kernel, dim3((batch + threads - 1) / threads), dim3(threads), 0, s, ratio, rid,
                    seq_lens, batch, plan_d, d_status);
}

namespace {

int launch_plan_prefill(PrefillPlanArgs a, cudaStream_t stream) {
  const uint32_t batch = a.batch;
  if (a.ratio != 4 && a.ratio != 128) return CKV_ERR_RATIO;
  if (batch > CKV_MAX_BATCH || a.num_q_tokens > CKV_MAX_TOKENS) return CKV_ERR_SIZE;
  if (a.cap_c > CKV_MAX_TOKENS + 1u || a.cap_w > CKV_MAX_TOKENS + 1u) return CKV_ERR_SIZE;
  if (a.d_counts == nullptr || (reinterpret_cast<uintptr_t>(a.d_counts) & 3u)) return CKV_ERR_POINTER;
  if (batch > 0 && (!a.rid || !a.seq_lens || !a.extend_lens)) return CKV_ERR_POINTER;
  if ((reinterpret_cast<uintptr_t>(a.rid) | reinterpret_cast<uintptr_t>(a.seq_lens) |
       reinterpret_cast<uintptr_t>(a.extend_lens)) & 7u)
    return CKV_ERR_POINTER;
  if (a.cap_c > 0 && !aligned16(a.plan_c)) return CKV_ERR_POINTER;
  if (a.online) {
    if (a.cap_w > 0 && !aligned16(a.units)) return CKV_ERR_POINTER;
  } else if (a.cap_w > 0 && (a.plan_w == nullptr || (reinterpret_cast<uintptr_t>(a.plan_w) & 7u))) {
    return CKV_ERR_POINTER;
  }
  const uint32_t work = std::max(a.cap_c, a.cap_w);
  uint32_t grid = (work + kPlanThreads - 1) / kPlanThreads;
  grid = std::max<uint32_t>(1, std::min<uint32_t>(grid, 2u * static_cast<uint32_t>(sm_count())));
  return launch_pdl(a.ratio == 4 ? plan_prefill_kernel<4> : plan_prefill_kernel<128>, dim3(grid), dim3(kPlanThreads),
                    0, stream, a);
}

// Paged arguments shared by both paged planners: C4 needs a mapping; C128
// state is request-scoped (c_plan.cuh compute_c128_loc) and ring_size must be
// 128, the only ring in which read_page_0 -- the page the C128 pooling reads
// (compressor_v2.py) -- is the page of the record's own window.
int check_paged(int ratio, const int32_t* r2t, int64_t stride, const int64_t* f2s, int32_t sps, int32_t ring) {
  if (ratio == 128) return ring == 128 ? CKV_OK : CKV_ERR_SIZE;
  if (ratio != 4) return CKV_ERR_RATIO;
  if (sps <= 0 || ring < 8 || ring % 4 != 0 || sps % ring != 0 || stride <= 0) return CKV_ERR_SIZE;
  if (r2t == nullptr || f2s == nullptr || (reinterpret_cast<uintptr_t>(r2t) & 3u) ||
      (reinterpret_cast<uintptr_t>(f2s) & 7u))
    return CKV_ERR_POINTER;
  return CKV_OK;
}

}  // namespace

int ckv_plan_prefill(int ratio, const int64_t* rid, const int64_t* seq_lens, const int64_t* extend_lens,
                     uint32_t batch, uint32_t num_q_tokens, uint32_t capacity_c, uint32_t capacity_w,
                     int pad_invalid, ckv_compress_plan_t* plan_c, ckv_write_plan_t* plan_w, uint32_t* d_counts,
                     uint32_t* d_status, ckv_stream_t stream) {
  PrefillPlanArgs a{};
  a.ratio = ratio;
  a.rid = rid;
  a.seq_lens = seq_lens;
  a.extend_lens = extend_lens;
  a.batch = batch;
  a.num_q_tokens = num_q_tokens;
  a.cap_c = capacity_c;
  a.cap_w = capacity_w;
  a.pad_invalid = pad_invalid;
  a.plan_c = plan_c;
  a.plan_w = plan_w;
  a.d_counts = d_counts;
  a.d_status = d_status;
  a.sps = 1;
  a.ring = 1;
  return launch_plan_prefill(a, reinterpret_cast<cudaStream_t>(stream));
}

int ckv_plan_online_prefill(const int64_t* rid, const int64_t* seq_lens, const int64_t* extend_lens,
                            uint32_t batch, uint32_t num_q_tokens, int64_t slot_offset, uint32_t capacity_u,
                            int pad_invalid, ckv_online_unit_t* units, uint32_t* d_counts, uint32_t* d_status,
                            ckv_stream_t stream) {
  PrefillPlanArgs a{};
  a.ratio = 128;
  a.rid = rid;
  a.seq_lens = seq_lens;
  a.extend_lens = extend_lens;
  a.batch = batch;
  a.num_q_tokens = num_q_tokens;
  a.cap_c = 0;
  a.cap_w = capacity_u;
  a.pad_invalid = pad_invalid;
  a.d_counts = d_counts;
  a.d_status = d_status;
  a.sps = 1;
  a.ring = 1;
  a.online = 1;
  a.slot_offset = slot_offset;
  a.units = units;
  return launch_plan_prefill(a, reinterpret_cast<cudaStream_t>(stream));
}

uint32_t ckv_capacity_online_units(uint32_t batch, uint32_t num_q_tokens) {
  const uint64_t u = static_cast<uint64_t>(num_q_tokens) / 128 + 2ull * batch;
  return static_cast<uint32_t>(std::min<uint64_t>(u, num_q_tokens));
}

int ckv_plan_prefill_paged(int ratio, const int64_t* rid, const int32_t* req_to_token, int64_t r2t_stride,
                           uint32_t num_reqs, const int64_t* full_to_state, uint64_t num_full_slots,
                           int32_t swa_page_size, int32_t ring_size, const int64_t* seq_lens,
                           const int64_t* extend_lens, uint32_t batch, uint32_t num_q_tokens, uint32_t capacity_c,
                           uint32_t capacity_w, int pad_invalid, ckv_compress_plan_t* plan_c,
                           ckv_write_plan_t* plan_w, uint32_t* d_counts, uint32_t* d_status, ckv_stream_t stream) {
  const int rc = check_paged(ratio, req_to_token, r2t_stride, full_to_state, swa_page_size, ring_size);
  if (rc) return rc;
  PrefillPlanArgs a{};
  a.ratio = ratio;
  a.rid = rid;
  a.seq_lens = seq_lens;
  a.extend_lens = extend_lens;
  a.batch = batch;
  a.num_q_tokens = num_q_tokens;
  a.cap_c = capacity_c;
  a.cap_w = capacity_w;
  a.pad_invalid = pad_invalid;
  a.plan_c = plan_c;
  a.plan_w = plan_w;
  a.d_counts = d_counts;
  a.d_status = d_status;
  a.paged = 1;
  a.r2t = req_to_token;
  a.r2t_stride = r2t_stride;
  a.num_reqs = num_reqs;
  a.f2s = full_to_state;
  a.num_full = num_full_slots;
  a.sps = swa_page_size;
  a.ring = ring_size;
  return launch_plan_prefill(a, reinterpret_cast<cudaStream_t>(stream));
}

int ckv_plan_decode_paged(int ratio, const int64_t* rid, const int32_t* req_to_token, int64_t r2t_stride,
                          uint32_t num_reqs, const int64_t* full_to_state, uint64_t num_full_slots,
                          int32_t swa_page_size, int32_t ring_size, const int64_t* seq_lens, uint32_t batch,
                          ckv_decode_plan_t* plan_d, ckv_decode_order_t* order, uint32_t* d_status,
                          ckv_stream_t stream) {
  const int rc = check_paged(ratio, req_to_token, r2t_stride, full_to_state, swa_page_size, ring_size);
  if (rc) return rc;
  if (ratio == 128) return ckv_plan_decode(ratio, rid, seq_lens, batch, plan_d, order, d_status, stream);
  if (batch == 0 && order == nullptr) return CKV_OK;
  if (batch > 0 && (!rid || !seq_lens || !aligned16(plan_d))) return CKV_ERR_POINTER;
  if ((reinterpret_cast<uintptr_t>(rid) | reinterpret_cast<uintptr_t>(seq_lens)) & 7u) return CKV_ERR_POINTER;
  DecodePagedArgs a{rid, seq_lens, batch, req_to_token, r2t_stride, num_reqs, full_to_state, num_full_slots,
                    swa_page_size, ring_size, plan_d, d_status};
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (order != nullptr) {
    if (reinterpret_cast<uintptr_t>(order) & 7u) return CKV_ERR_POINTER;
    if (batch <= kPlanThreads)
      return launch_pdl(plan_decode_paged_ordered_kernel<1>, dim3(1), dim3(kPlanThreads), 0, s, a, order);
    return launch_pdl(plan_decode_paged_ordered_kernel<4>, dim3(1), dim3(kPlanThreads), 0, s, a, order);
  }
  const uint32_t threads = 256;
  return launch_pdl(plan_decode_paged_kernel, dim3((batch + threads - 1) / threads), dim3(threads), 0, s, a);
}

uint32_t ckv_capacity_write_paged(int ratio, uint32_t batch, uint32_t num_q_tokens, int32_t swa_page_size) {
  if (ratio != 4 || swa_page_size <= 0) return ckv_capacity_write(ratio, batch, num_q_tokens);
  const uint64_t w = static_cast<uint64_t>(batch) * 7 +
                     4ull * (static_cast<uint64_t>(num_q_tokens) / static_cast<uint64_t>(swa_page_size) + batch);
  return static_cast<uint32_t>(std::min<uint64_t>(w, num_q_tokens));
}

const char* ckv_error_string(int code) {
  switch (code) {
    case CKV_OK: return "ok";
    case CKV_ERR_RATIO: return "ratio must be 4 or 128";
    case CKV_ERR_HEAD_DIM: return "head_dim must be a positive multiple of 128 and at most 1024";
    case CKV_ERR_SIZE: return "a batch, token count or capacity is out of range";
    case CKV_ERR_POINTER: return "a required pointer is NULL or misaligned";
    case CKV_ERR_DTYPE: return "unsupported dtype or layout";
    case CKV_ERR_LAUNCH: return "CUDA launch failed";
    default: return "unknown ckv error";
  }
}

int ckv_version(void) { return 220; }

}  // extern "C"
