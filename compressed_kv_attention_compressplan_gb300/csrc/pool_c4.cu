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
// Prefill: a producer warp stages each record's window in shared memory with
// two tensor-map copies (see c4_pool_prefill_staged_kernel); consumer threads
// own 16-byte channel chunks (8 bf16 or 4 fp32 channels).  Small steps load
// the windows directly instead, one thread per record and chunk
// (c4_pool_prefill_direct_kernel).  Decode: one thread
// per (row, 4 channels) with direct loads.  The window is small enough that
// the fp32 safe softmax runs entirely in registers.
#include <algorithm>
#include <atomic>
#include <cstring>

#include "async_copy.cuh"
#include "common.cuh"
#include "launch.h"

namespace ckv {
namespace {

template <typename TIn>
struct C4Vec {
  static constexpr int VEC = 16 / static_cast<int>(sizeof(TIn));  // channels per 16-byte chunk
};

// The decode's unit: four channels of one row (8 bytes of bf16, 16 of fp32).
// A decode batch is small, so its rows spread over few threads per SM, and
// one unit's reduction is a chain of dependent instructions per channel: four
// channels per thread halve that chain for bf16 and double the warps that
// hide its latency.
template <typename TIn>
struct C4DecVec;
template <>
struct C4DecVec<float> {
  using V = uint4;
};
template <>
struct C4DecVec<__nv_bfloat16> {
  using V = uint2;
};
constexpr int kC4DecVec = 4;

__device__ __forceinline__ uint2 ld_stream8(const void* p) {
  uint2 v;
  asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
  return v;
}

template <typename V>
__device__ __forceinline__ V ld_stream_v(const void* p);
template <>
__device__ __forceinline__ uint4 ld_stream_v<uint4>(const void* p) { return ld_stream16(p); }
template <>
__device__ __forceinline__ uint2 ld_stream_v<uint2>(const void* p) { return ld_stream8(p); }

template <typename V>
__device__ __forceinline__ V ld_cached_v(const void* p) { return __ldg(reinterpret_cast<const V*>(p)); }

template <typename V>
__device__ __forceinline__ void st_v(void* p, const V& v) { *reinterpret_cast<V*>(p) = v; }

template <typename V>
__device__ __forceinline__ V zero_v();
template <>
__device__ __forceinline__ uint4 zero_v<uint4>() { return make_uint4(0, 0, 0, 0); }
template <>
__device__ __forceinline__ uint2 zero_v<uint2>() { return make_uint2(0, 0); }

// Element j of a vector of TIn as fp32.
template <typename TIn>
__device__ __forceinline__ float unpack_v(const uint4& v, int j) { return unpack<TIn>(v, j); }
template <typename TIn>
__device__ __forceinline__ float unpack_v(const uint2& v, int j) {
  const uint32_t w = sizeof(TIn) == 2 ? ((j >> 1) == 0 ? v.x : v.y) : (j == 0 ? v.x : v.y);
  return sizeof(TIn) == 2 ? ((j & 1) ? bf16hi(w) : bf16lo(w)) : __uint_as_float(w);
}

// One 4-D tensor-map box (channel 0, block q0, both parts, rows from `row`)
// -> shared memory, completing on `bar`.
__device__ __forceinline__ void tma_box4_g2s(uint32_t dst, const CUtensorMap* map, int q0, int row, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, %5}], "
      "[%6];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(0), "r"(q0), "r"(0), "r"(row), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

__device__ __forceinline__ void prefetch_map(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// The C4 window pool for VEC channels.  Entries below `first` are masked.
// (Scalar form: with 16 kv/score vectors live, the packed fp32x2 form of the
// same operations needs more registers than this kernel can spare.)
template <typename TIn, int VEC, typename V>
__device__ __forceinline__ void c4_pool_chunk(const V (&kv)[8], const V (&sc)[8], const V (&ap)[8], int first,
                                              float (&res)[VEC]) {
#pragma unroll
  for (int j = 0; j < VEC; ++j) {
    float s[8];
    float m = -INFINITY;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      s[i] = score_plus_bias(unpack_v<TIn>(sc[i], j), unpack_v<TIn>(ap[i], j));
      if (i >= first) m = fmaxf(m, s[i]);
    }
    const float nml = neg_max_log2e(m);
    PoolAcc acc;
    acc.init();
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      if (i >= first) acc.add(unpack_v<TIn>(kv[i], j), weight_of(s[i], nml));
    }
    res[j] = finish(acc.a, acc.l);
  }
}

// Prefill, staged by the TMA engine.  A C4 row, | kv-overlap | kv |
// score-overlap | score |, is viewed as a 4-D tensor (channel within a block
// of c4_block(hd) channels, block within a part -- the overlap quarter
// then the main quarter, part -- kv or score, row), so that the overlap
// halves of four consecutive rows (window entries 0..3) or their main halves
// (entries 4..7) are ONE box: a record whose window lies in the input is two
// copies.  Entries held in the ring come from the state through the same view
// (a box of 4 rows when a whole group is in the state, else one row at a
// time).  A producer warp issues the copies of C4Stage::recs(hd) consecutive
// records per stage into a ring; the window of record r of a stage sits at
// [entry][kv | score][head_dim] and consumer thread t owns 16-byte channel
// chunk t % chunks of record t / chunks, running the same c4_pool_chunk as the
// other C4 kernels (the rows are bit-identical to theirs).  Pseudo-record
// num_c (token layout) zeroes the rows after the last compress row.
constexpr int kC4StageBudget = 192 * 1024;  // ring bytes per CTA

// Channels per block of the 4-D view: it must divide head_dim (a multiple of
// 128) and stay within a box's 256-element limit.
__host__ __device__ constexpr int c4_block(int hd) { return hd % 256 == 0 ? 256 : 128; }

template <typename TIn>
struct C4Stage {
  __host__ __device__ static int chunks(int hd) { return hd / C4Vec<TIn>::VEC; }
  // records per stage: enough that a stage keeps 256 consumer threads busy
  __host__ __device__ static int recs(int hd) { return chunks(hd) >= 256 ? 1 : 256 / chunks(hd); }
  __host__ __device__ static int active(int hd) { return recs(hd) * chunks(hd); }
  // whole warps: the producer must be one warp of its own
  __host__ __device__ static int consumers(int hd) { return (active(hd) + 31) / 32 * 32; }
  __host__ __device__ static uint32_t bytes(int hd) {
    return static_cast<uint32_t>(recs(hd)) * 16u * static_cast<uint32_t>(hd) * sizeof(TIn);
  }
  __host__ __device__ static int stages(int hd) {
    const int n = kC4StageBudget / static_cast<int>(bytes(hd));
    return n < 2 ? 2 : n > 8 ? 8 : n;
  }
  // Small steps: half the records per stage in half the ring, so that two
  // CTAs fit on an SM and a stage's reductions run on half as many records.
  __host__ __device__ static int recs_small(int hd) { return recs(hd) >= 2 ? recs(hd) / 2 : recs(hd); }
  __host__ __device__ static uint32_t bytes_small(int hd) {
    return static_cast<uint32_t>(recs_small(hd)) * 16u * static_cast<uint32_t>(hd) * sizeof(TIn);
  }
  __host__ __device__ static int stages_small(int hd) {
    const int n = kC4StageBudget / 2 / static_cast<int>(bytes_small(hd));
    return n < 2 ? 2 : n > 8 ? 8 : n;
  }
};

// The four views: input and state, boxes of 4 rows and of 1 row.
struct C4Maps {
  CUtensorMap in4, in1, st4, st1;
};

// A compress record as the staged kernel uses it (false: padding, or a record
// pointing outside the state / input, which also sets `bad`).
struct C4Rec {
  uint32_t ragged;
  int bl, first;
  int64_t rp0, rp1;
};

__device__ __forceinline__ ckv_compress_plan_t c4_load_record(const PoolArgs& a, uint32_t e, uint32_t num_c) {
  if (e < num_c) return load_plan_c(a.plan_c + e);
  ckv_compress_plan_t P;
  P.seq_len = kInvalidU32;
  P.ragged_bl = kInvalidU32;
  P.read_page_0 = P.read_page_1 = -1;
  return P;
}

__device__ __forceinline__ bool c4_record(const PoolArgs& a, const ckv_compress_plan_t& P, C4Rec& r, bool& bad) {
  bad = false;
  if (plan_c_invalid(P)) return false;
  r.ragged = P.ragged_bl & CKV_RAGGED_MASK;
  r.bl = static_cast<int>(P.ragged_bl >> CKV_BUFFER_LEN_SHIFT);
  r.first = P.seq_len == 4 ? 4 : 0;
  r.rp0 = P.read_page_0;
  r.rp1 = P.read_page_1;
  bool ok = r.ragged < a.num_q_tokens && r.bl <= 7 && static_cast<int64_t>(r.ragged) - 7 + r.bl >= 0;
  if (r.bl > r.first && r.first < 4) ok = ok && r.rp0 >= 0 && static_cast<uint64_t>(r.rp0) * 4 + 3 < a.state_rows;
  if (r.bl > 4) ok = ok && r.rp1 >= 0 && static_cast<uint64_t>(r.rp1) * 4 + 3 < a.state_rows;
  bad = !ok;
  return ok;
}

// Issues the copies of record r's window into `win` ([8][2][hd] elements);
// returns their bytes.  q = blocks per quarter.
template <typename TIn>
__device__ __forceinline__ uint32_t c4_issue_window(const C4Maps& m, const C4Rec& r, int hd, int q, TIn* win,
                                                    uint32_t bar, bool issue) {
  const uint32_t row_bytes = 2u * static_cast<uint32_t>(hd) * sizeof(TIn);  // one entry: kv + score halves
  uint32_t bytes = 0;
  for (int p = 0; p < 2; ++p) {
    const int i0 = 4 * p;
    if (p == 0 && r.first == 4) continue;  // the first group has no previous group
    const int q0 = p == 0 ? 0 : q;
    const int page_row = static_cast<int>((p == 0 ? r.rp0 : r.rp1) * 4);
    if (i0 >= r.bl) {  // four input rows
      if (issue)
        tma_box4_g2s(smem_addr(win + static_cast<size_t>(2 * i0) * hd), &m.in4, q0,
                     static_cast<int>(r.ragged) - 7 + i0, bar);
      bytes += 4 * row_bytes;
    } else if (i0 + 4 <= r.bl) {  // a whole 4-slot page of the ring
      if (issue) tma_box4_g2s(smem_addr(win + static_cast<size_t>(2 * i0) * hd), &m.st4, q0, page_row, bar);
      bytes += 4 * row_bytes;
    } else {
      for (int i = i0; i < i0 + 4; ++i) {
        if (issue) {
          if (i < r.bl)
            tma_box4_g2s(smem_addr(win + static_cast<size_t>(2 * i) * hd), &m.st1, q0, page_row + (i & 3), bar);
          else
            tma_box4_g2s(smem_addr(win + static_cast<size_t>(2 * i) * hd), &m.in1, q0,
                         static_cast<int>(r.ragged) - 7 + i, bar);
        }
        bytes += row_bytes;
      }
    }
  }
  return bytes;
}

template <typename TIn, typename TOut, bool kShortWaits, bool kSmall>
__global__ __launch_bounds__(288, 1) void c4_pool_prefill_staged_kernel(const PoolArgs a,
                                                                        const __grid_constant__ C4Maps maps) {
  using S = C4Stage<TIn>;
  constexpr int VEC = C4Vec<TIn>::VEC;
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t full_bar[8];
  __shared__ __align__(8) uint64_t empty_bar[8];
  __shared__ volatile int abort_flag;
  const int hd = a.head_dim;
  const int q = hd / c4_block(hd);
  const int chunks = S::chunks(hd);
  const int R = kSmall ? S::recs_small(hd) : S::recs(hd);
  const int NCT = (R * chunks + 31) / 32 * 32;
  const int NS = kSmall ? S::stages_small(hd) : S::stages(hd);
  const bool active = threadIdx.x < R * chunks;
  const uint32_t stage_bytes = kSmall ? S::bytes_small(hd) : S::bytes(hd);
  const int t = threadIdx.x;
  if (t == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(smem_addr(&full_bar[s]), 1);
      mbar_init(smem_addr(&empty_bar[s]), static_cast<uint32_t>(NCT / 32));
    }
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (a.ext_hint != nullptr) {
    // Small steps only (see the host): while the planner runs, into L2 the
    // state halves that each request's first window reads (legacy ring rows
    // rid * 8 + position % 8; entries 0..3 take the overlap halves, 4..7 the
    // main ones), one thread per request.  Line prefetches, not bulk ones: the
    // copy engine takes bulk prefetches in order with the stage copies, and a
    // thousand 1 KB ones ahead of them held the first stage back by ~8 us.
    // (Prefetching the input too only moved time from the pool to the write.)
    // The hints are the planner's own inputs, read before the dependency wait:
    // they only steer prefetches.
    const uint32_t half = static_cast<uint32_t>(hd) * sizeof(TIn);
    const uint32_t row_bytes = 4u * half;
    const uint8_t* st = static_cast<const uint8_t*>(a.state);
    for (uint32_t b = blockIdx.x + static_cast<uint32_t>(t) * gridDim.x; b < a.hint_batch;
         b += blockDim.x * gridDim.x) {
      int64_t sl, el, rid;
      asm volatile("ld.global.u64 %0, [%1];" : "=l"(sl) : "l"(a.seq_hint + b));
      asm volatile("ld.global.u64 %0, [%1];" : "=l"(el) : "l"(a.ext_hint + b));
      asm volatile("ld.global.u64 %0, [%1];" : "=l"(rid) : "l"(a.rid_hint + b));
      const int64_t pl = sl - el;
      if (el > 0 && pl > 0 && sl / 4 > pl / 4 && rid >= 0 && rid < (int64_t{1} << 48) &&
          static_cast<uint64_t>(rid) * 8 + 7 < a.state_rows) {
        const int64_t p = pl / 4 * 4 + 3;  // the request's first event
        for (int i = p == 3 ? 4 : 0; i < 8 && p - 7 + i < pl; ++i) {
          const uint8_t* row = st + static_cast<size_t>(rid * 8 + (p - 7 + i) % 8) * row_bytes;
          for (uint32_t o = 0; o < half; o += 128) {
            prefetch_l2(row + (i < 4 ? 0 : half) + o);
            prefetch_l2(row + (i < 4 ? 2 : 3) * half + o);
          }
        }
      }
    }
  }
  pdl_wait();
  pdl_release();
  const bool token = a.out_layout == CKV_OUT_TOKEN;
  const uint32_t num_c = count_or_capacity(a.d_counts, 0, a.capacity);
  const uint32_t n_rec = num_c + (token ? 1u : 0u);  // + the tail pseudo-record
  const uint32_t n_grp = (n_rec + R - 1) / R;

  if (t >= NCT) {
    // ---------------- producer warp: lane r issues record r of the stage
    const int lane = t - NCT;
    if (lane < 4) prefetch_map(lane == 0 ? &maps.in4 : lane == 1 ? &maps.in1 : lane == 2 ? &maps.st4 : &maps.st1);
    uint32_t g = 0;
    // each lane's record of the next group is requested one group ahead
    ckv_compress_plan_t nxt = c4_load_record(a, blockIdx.x * R + lane, lane < R ? num_c : 0u);
    for (uint32_t grp = blockIdx.x; grp < n_grp && !__any_sync(0xFFFFFFFFu, abort_flag != 0);
         grp += gridDim.x, ++g) {
      const ckv_compress_plan_t cur = nxt;
      nxt = c4_load_record(a, (grp + gridDim.x) * R + lane, lane < R ? num_c : 0u);
      const int stage = static_cast<int>(g % NS);
      if (!warp_wait_for<kShortWaits>(smem_addr(&empty_bar[stage]), ((g / NS) & 1u) ^ 1u, a.wait_ns)) {
        if (lane == 0) {
          status_or(a.d_status, CKV_STATUS_TIMEOUT);
          abort_flag = 1;
        }
        break;
      }
      C4Rec rec;
      bool bad;
      const bool mine = lane < R && c4_record(a, cur, rec, bad);
      TIn* win = reinterpret_cast<TIn*>(smem + static_cast<size_t>(stage) * stage_bytes) +
                 static_cast<size_t>(lane) * 16 * hd;
      const uint32_t bar = smem_addr(&full_bar[stage]);
      uint32_t total = mine ? c4_issue_window<TIn>(maps, rec, hd, q, win, bar, false) : 0u;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) total += __shfl_xor_sync(0xFFFFFFFFu, total, off);
      if (lane == 0) mbar_arrive_expect_tx(bar, total);  // announced before any copy is issued
      __syncwarp();
      if (mine) c4_issue_window<TIn>(maps, rec, hd, q, win, bar, true);
    }
    // the last NS stages issued have landed before the CTA can exit
    for (uint32_t h = g > static_cast<uint32_t>(NS) ? g - NS : 0u; h < g; ++h)
      mbar_wait_bounded(smem_addr(&full_bar[h % NS]), (h / NS) & 1u, kWaitLimitNs);
    return;
  }

  // ---------------- consumers
  const int r = t / chunks;
  const int ch = t % chunks;
  const int c0 = ch * VEC;
  const int lane = t & 31;
  TOut* out = static_cast<TOut*>(a.out);
  const TIn* ape = static_cast<const TIn*>(a.ape);
  uint4 ap[8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
    ap[i] = active ? ld_cached16(ape + static_cast<size_t>(i) * hd + c0) : make_uint4(0, 0, 0, 0);
  uint32_t g = 0;
  // this thread's record of the next group (and the one before it, for the
  // zero rows of the token layout) are requested one group ahead
  const uint32_t num_c_mine = active ? num_c : 0u;
  ckv_compress_plan_t nxt = c4_load_record(a, blockIdx.x * R + r, num_c_mine);
  ckv_compress_plan_t nxt_prev = c4_load_record(a, blockIdx.x * R + r - 1, blockIdx.x * R + r > 0 ? num_c_mine : 0u);
  for (uint32_t grp = blockIdx.x; grp < n_grp; grp += gridDim.x, ++g) {
    const ckv_compress_plan_t cur = nxt, cur_prev = nxt_prev;
    const uint32_t en = (grp + gridDim.x) * R + r;
    nxt = c4_load_record(a, en, num_c_mine);
    nxt_prev = c4_load_record(a, en - 1, num_c_mine);
    const int stage = static_cast<int>(g % NS);
    if (!warp_wait_for<kShortWaits>(smem_addr(&full_bar[stage]), (g / NS) & 1u, a.wait_ns)) {
      status_or(a.d_status, CKV_STATUS_TIMEOUT);
      abort_flag = 1;
      break;
    }
    const uint32_t e = grp * R + r;
    if (!active) {
    } else if (e < num_c) {
      C4Rec rec;
      bool bad;
      if (c4_record(a, cur, rec, bad)) {
        const TIn* base = reinterpret_cast<const TIn*>(smem + static_cast<size_t>(stage) * stage_bytes) +
                          static_cast<size_t>(r) * 16 * hd + c0;
        uint4 kv[8], sc[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          if (i < rec.first) {
            kv[i] = sc[i] = make_uint4(0, 0, 0, 0);
          } else {
            kv[i] = *reinterpret_cast<const uint4*>(base + static_cast<size_t>(2 * i) * hd);
            sc[i] = *reinterpret_cast<const uint4*>(base + static_cast<size_t>(2 * i + 1) * hd);
          }
        }
        float res[VEC];
        c4_pool_chunk<TIn, VEC>(kv, sc, ap, rec.first, res);
        const size_t orow = token ? rec.ragged : e;
        store_row_chunk<TOut, VEC>(out + orow * hd + c0, res);
        if (token) {  // zero the rows between the previous compress row and this one
          int64_t prev = -1;
          if (e > 0)
            prev = plan_c_invalid(cur_prev) ? static_cast<int64_t>(rec.ragged)
                                            : static_cast<int64_t>(cur_prev.ragged_bl & CKV_RAGGED_MASK);
          for (int64_t row = prev + 1; row < static_cast<int64_t>(rec.ragged); ++row)
            store_zero_chunk<TOut, VEC>(out + static_cast<size_t>(row) * hd + c0);
        }
      } else if (bad && ch == 0) {
        status_or(a.d_status, CKV_STATUS_BAD_INDEX);
      }
    } else if (token && e == num_c) {  // rows after the last compress row
      int64_t last = -1;
      if (num_c > 0) {
        const ckv_compress_plan_t Q = load_plan_c(a.plan_c + num_c - 1);
        last = plan_c_invalid(Q) ? static_cast<int64_t>(a.num_q_tokens)
                                 : static_cast<int64_t>(Q.ragged_bl & CKV_RAGGED_MASK);
      }
      for (int64_t row = last + 1; row < static_cast<int64_t>(a.num_q_tokens); ++row)
        store_zero_chunk<TOut, VEC>(out + static_cast<size_t>(row) * hd + c0);
    }
    // this warp no longer reads the stage
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_addr(&empty_bar[stage]));
  }
}

// Small steps, direct loads: one thread per (record, 16-byte channel chunk),
// the grid one resident wave.  A thread requests its record (and the one
// before it, for the zero rows of the token layout) together with the count
// and the ape chunks, then its 16 window vectors at once, so a record costs
// two memory round trips after the dependency wait; the staged kernel's chain
// (count, record, copies issued, copies landed, stage handed over) is longer
// than a whole launch of a step of a few thousand records takes this way.
// Same c4_pool_chunk, so the rows are bit-identical to the other C4 kernels'.
constexpr int kC4DirectThreads = 128;

template <typename TIn, typename TOut>
__global__ __launch_bounds__(kC4DirectThreads) void c4_pool_prefill_direct_kernel(const PoolArgs a, uint32_t chunks,
                                                                                 uint32_t cap_units) {
  constexpr int VEC = C4Vec<TIn>::VEC;
  const int hd = a.head_dim;
  const size_t width = 4 * static_cast<size_t>(hd);
  const TIn* state = static_cast<const TIn*>(a.state);
  const TIn* input = static_cast<const TIn*>(a.input);
  const TIn* ape = static_cast<const TIn*>(a.ape);
  TOut* out = static_cast<TOut*>(a.out);
  const uint32_t tid = blockIdx.x * blockDim.x + threadIdx.x;
  const uint32_t stride = gridDim.x * blockDim.x;
  if (a.ext_hint != nullptr) {
    // As in the staged kernel: the state halves of each request's first
    // window into L2 while the planner runs, one 128-byte line of one entry's
    // kv and score halves per item.  Only prefetches follow from the hints.
    const uint32_t half = static_cast<uint32_t>(hd) * sizeof(TIn);
    const uint32_t lines = half / 128;
    const uint8_t* st = static_cast<const uint8_t*>(a.state);
    const uint64_t items = static_cast<uint64_t>(a.hint_batch) * 8 * lines;
    for (uint64_t k = tid; k < items; k += stride) {
      const uint32_t b = static_cast<uint32_t>(k / (8 * lines));
      const int i = static_cast<int>((k / lines) % 8);
      const uint32_t o = static_cast<uint32_t>(k % lines) * 128;
      int64_t sl, el, rid;
      asm volatile("ld.global.u64 %0, [%1];" : "=l"(sl) : "l"(a.seq_hint + b));
      asm volatile("ld.global.u64 %0, [%1];" : "=l"(el) : "l"(a.ext_hint + b));
      asm volatile("ld.global.u64 %0, [%1];" : "=l"(rid) : "l"(a.rid_hint + b));
      const int64_t pl = sl - el;
      if (el > 0 && pl > 0 && sl / 4 > pl / 4 && rid >= 0 && rid < (int64_t{1} << 48) &&
          static_cast<uint64_t>(rid) * 8 + 7 < a.state_rows) {
        const int64_t p = pl / 4 * 4 + 3;  // the request's first event
        if (i >= (p == 3 ? 4 : 0) && p - 7 + i < pl) {
          const uint8_t* row = st + static_cast<size_t>(rid * 8 + (p - 7 + i) % 8) * 4 * half;
          prefetch_l2(row + (i < 4 ? 0 : half) + o);
          prefetch_l2(row + (i < 4 ? 2 : 3) * half + o);
        }
      }
    }
  }
  pdl_wait();
  pdl_release();
  const bool token = a.out_layout == CKV_OUT_TOKEN;
  const uint32_t num_c = count_or_capacity(a.d_counts, 0, a.capacity);
  for (uint32_t u = tid; u < cap_units; u += stride) {
    const uint32_t e = u / chunks;
    const int c0 = static_cast<int>(u % chunks) * VEC;
    // requested before num_c is known (both slots exist: e - 1 < e < capacity)
    ckv_compress_plan_t P, Pp;
    P.seq_len = Pp.seq_len = kInvalidU32;
    if (e < a.capacity) P = load_plan_c(a.plan_c + e);
    if (e > 0 && e - 1 < a.capacity) Pp = load_plan_c(a.plan_c + e - 1);
    uint4 ap[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) ap[i] = ld_cached16(ape + static_cast<size_t>(i) * hd + c0);
    if (e > num_c || (e == num_c && !token)) break;  // u only grows
    if (e == num_c) {  // token layout: the rows after the last compress row
      const int64_t last = num_c == 0 ? -1
                           : plan_c_invalid(Pp) ? static_cast<int64_t>(a.num_q_tokens)
                                                : static_cast<int64_t>(Pp.ragged_bl & CKV_RAGGED_MASK);
      for (int64_t row = last + 1; row < static_cast<int64_t>(a.num_q_tokens); ++row)
        store_zero_chunk<TOut, VEC>(out + static_cast<size_t>(row) * hd + c0);
      continue;
    }
    C4Rec rec;
    bool bad;
    if (!c4_record(a, P, rec, bad)) {
      if (bad && c0 == 0) status_or(a.d_status, CKV_STATUS_BAD_INDEX);
      continue;
    }
    uint4 kv[8], sc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      kv[i] = sc[i] = make_uint4(0, 0, 0, 0);
      if (i >= rec.first) {
        // entries held in the ring were checked inside the state by c4_record
        const TIn* row = i < rec.bl ? state + static_cast<size_t>((i < 4 ? rec.rp0 : rec.rp1) * 4 + (i & 3)) * width
                                    : input + (static_cast<size_t>(rec.ragged) + i - 7) * width;
        kv[i] = ld_stream16(row + (i < 4 ? 0 : hd) + c0);
        sc[i] = ld_stream16(row + (i < 4 ? 2 * hd : 3 * hd) + c0);
      }
    }
    float res[VEC];
    c4_pool_chunk<TIn, VEC>(kv, sc, ap, rec.first, res);
    store_row_chunk<TOut, VEC>(out + (token ? static_cast<size_t>(rec.ragged) : e) * hd + c0, res);
    if (token) {  // zero the rows between the previous compress row and this one
      int64_t prev = -1;
      if (e > 0)
        prev = plan_c_invalid(Pp) ? static_cast<int64_t>(rec.ragged)
                                  : static_cast<int64_t>(Pp.ragged_bl & CKV_RAGGED_MASK);
      for (int64_t row = prev + 1; row < static_cast<int64_t>(rec.ragged); ++row)
        store_zero_chunk<TOut, VEC>(out + static_cast<size_t>(row) * hd + c0);
    }
  }
}

// Decode: one unit per (row, 4 channels).  The new token's row is written to
// its ring slot; at a group boundary the window's first 7 entries come from
// the ring (none of them is the slot being written) and entry 7 is the new
// token.  The new token's unit and the ape units do not depend on the plan
// record, so they are requested together with it, and so is the window that
// the rid / seq_lens hints name when given: a boundary row then costs one
// memory round trip when the record agrees with the hints (two otherwise),
// any other row one.
// Blocks of at most this many threads, sized on the host so that every SM
// gets the same number of blocks (see launch_decode_t).
constexpr int kC4DecodeMaxThreads = 256;

template <typename TIn, typename TOut>
__global__ __launch_bounds__(kC4DecodeMaxThreads) void c4_decode_kernel(const PoolArgs a, uint32_t chunks,
                                                                     uint32_t units) {
  using V = typename C4DecVec<TIn>::V;
  constexpr int VEC = kC4DecVec;
  constexpr int kLineUnits = 128 / static_cast<int>(sizeof(V));  // units per 128-byte line
  const uint32_t u = blockIdx.x * blockDim.x + threadIdx.x;
  const int hd = a.head_dim;
  const size_t width = 4 * static_cast<size_t>(hd);
  TIn* state = static_cast<TIn*>(a.state_mut);
  const TIn* input = static_cast<const TIn*>(a.input);
  const TIn* ape = static_cast<const TIn*>(a.ape);
  TOut* out = static_cast<TOut*>(a.out);
  const uint32_t b = u / chunks;
  const uint32_t ch = u % chunks;
  const int c0 = static_cast<int>(ch) * VEC;
  bool h_ok = false;  // the hints name a boundary row whose legacy ring is inside the state
  int64_t h_sl = 0, h_rid = 0;
  if (u < units) {
    // While the previous kernel finishes: this row's plan record, its new
    // token and, from the rid / seq_lens hints (legacy ring rows rid * 8 +
    // position % 8), the ring lines its window reads, into L2 (one thread per
    // 128-byte line).  Nothing read before the dependency wait is used after
    // it except through the check below, so a stale hint only costs bandwidth.
    const bool line = ch % kLineUnits == 0;
    const TIn* src = input + static_cast<size_t>(b) * width + c0;
    if (ch == 0) prefetch_l2(a.plan_d + b);
    if (line) {
      prefetch_l2(src);
      prefetch_l2(src + hd);
      prefetch_l2(src + 2 * hd);
      prefetch_l2(src + 3 * hd);
    }
    if (a.seq_hint != nullptr) {
      int64_t sl, rid;
      asm volatile("ld.global.u64 %0, [%1];" : "=l"(sl) : "l"(a.seq_hint + b));
      asm volatile("ld.global.u64 %0, [%1];" : "=l"(rid) : "l"(a.rid_hint + b));
      if (sl >= 4 && sl % 4 == 0 && rid >= 0 && static_cast<uint64_t>(rid) * 8 + 7 < a.state_rows) {
        h_ok = true;
        h_sl = sl;
        h_rid = rid;
        if (line) {
          const int64_t p = sl - 1;
          for (int i = sl == 4 ? 4 : 0; i < 7; ++i) {
            const int64_t q = p - 7 + i;  // the position of window entry i
            const TIn* row = state + static_cast<size_t>(rid * 8 + q % 8) * width;
            prefetch_l2(row + (i < 4 ? 0 : hd) + c0);
            prefetch_l2(row + (i < 4 ? 2 * hd : 3 * hd) + c0);
          }
        }
      }
    }
  }
  pdl_wait();
  pdl_release();
  if (u >= units) return;
  TOut* orow = out + static_cast<size_t>(b) * hd + c0;

  const ckv_decode_plan_t P = load_plan_d(a.plan_d + b);
  const TIn* src = input + static_cast<size_t>(b) * width + c0;  // row b of the input always exists
  const V kv_ovl = ld_stream_v<V>(src), kv_main = ld_stream_v<V>(src + hd);
  const V sc_ovl = ld_stream_v<V>(src + 2 * hd), sc_main = ld_stream_v<V>(src + 3 * hd);
  V ap[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) ap[i] = ld_cached_v<V>(ape + static_cast<size_t>(i) * hd + c0);
  // The window as the hints name it, requested together with the record (one
  // round trip instead of two); used below only if the record names the same
  // rows, whose slots no row of this step writes.
  const int h_first = h_sl == 4 ? 4 : 0;
  V kv[8], sc[8];
#pragma unroll
  for (int i = 0; i < 7; ++i) {
    kv[i] = sc[i] = zero_v<V>();
    if (h_ok && i >= h_first) {
      const TIn* row = state + static_cast<size_t>(h_rid * 8 + (h_sl - 8 + i) % 8) * width;
      kv[i] = ld_stream_v<V>(row + (i < 4 ? 0 : hd) + c0);
      sc[i] = ld_stream_v<V>(row + (i < 4 ? 2 * hd : 3 * hd) + c0);
    }
  }
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
  st_v<V>(dst, kv_ovl);
  st_v<V>(dst + hd, kv_main);
  st_v<V>(dst + 2 * hd, sc_ovl);
  st_v<V>(dst + 3 * hd, sc_main);
  if (!boundary) {
    store_zero_chunk<TOut, VEC>(orow);
    return;
  }
  const int first = P.seq_len == 4 ? 4 : 0;
  bool same = h_ok && h_sl == static_cast<int64_t>(P.seq_len);
#pragma unroll
  for (int i = 0; i < 7; ++i)
    if (i >= first) same = same && (i < 4 ? rp0 : rp1) * 4 + (i & 3) == h_rid * 8 + (h_sl - 8 + i) % 8;
  if (!same) {  // the rows the record names
#pragma unroll
    for (int i = 0; i < 7; ++i) {
      if (i < first) {
        kv[i] = sc[i] = zero_v<V>();
        continue;
      }
      const TIn* row = state + static_cast<size_t>((i < 4 ? rp0 : rp1) * 4 + (i & 3)) * width;
      kv[i] = ld_stream_v<V>(row + (i < 4 ? 0 : hd) + c0);
      sc[i] = ld_stream_v<V>(row + (i < 4 ? 2 * hd : 3 * hd) + c0);
    }
  }
  kv[7] = kv_main;
  sc[7] = sc_main;
  float res[VEC];
  c4_pool_chunk<TIn, VEC>(kv, sc, ap, first, res);
  store_row_chunk<TOut, VEC>(orow, res);
}

// Decode fused with RMSNorm + RoPE + store (ckv_compress_decode_norm_rope_store):
// the decode above, whose pooled row (fp32, or +0.0 off a group boundary)
// goes through y_c = x_c * w_c / sqrt(mean(x^2) + eps), the RoPE pairs of the
// last rope_dim channels at table row max(seq_len - 4, 0), and straight into
// cache row out_loc[b] -- the composition of ckv_compress_decode (fp32 out)
// and ckv_norm_rope_store_decode without the pooled rows in between.  A row's
// units are consecutive threads of one block (a block of 128 threads holds
// 128 / U rows of U = head_dim / 4 units, or one row when U does not divide
// 128): the sum of squares is a warp butterfly, then a sum over the row's
// warps in shared memory, in warp order.
template <typename TIn>
__global__ __launch_bounds__(256) void c4_decode_norm_kernel(const PoolArgs a, const DecodeNormArgs n, uint32_t chunks,
                                                             uint32_t units) {
  using V = typename C4DecVec<TIn>::V;
  constexpr int VEC = kC4DecVec;
  constexpr int kLineUnits = 128 / static_cast<int>(sizeof(V));
  __shared__ float s_part[8];
  const uint32_t u = blockIdx.x * blockDim.x + threadIdx.x;
  const bool live = u < units;
  const int hd = a.head_dim;
  const size_t width = 4 * static_cast<size_t>(hd);
  TIn* state = static_cast<TIn*>(a.state_mut);
  const TIn* input = static_cast<const TIn*>(a.input);
  const TIn* ape = static_cast<const TIn*>(a.ape);
  const uint32_t b = u / chunks;
  const uint32_t ch = u % chunks;
  const int c0 = static_cast<int>(ch) * VEC;
  bool h_ok = false;
  int64_t h_sl = 0, h_rid = 0;
  if (live) {  // L2 prefetches from the hints, as in c4_decode_kernel
    const bool line = ch % kLineUnits == 0;
    const TIn* src = input + static_cast<size_t>(b) * width + c0;
    if (ch == 0) prefetch_l2(a.plan_d + b);
    if (line) {
      prefetch_l2(src);
      prefetch_l2(src + hd);
      prefetch_l2(src + 2 * hd);
      prefetch_l2(src + 3 * hd);
    }
    if (a.seq_hint != nullptr) {
      int64_t sl, rid;
      asm volatile("ld.global.u64 %0, [%1];" : "=l"(sl) : "l"(a.seq_hint + b));
      asm volatile("ld.global.u64 %0, [%1];" : "=l"(rid) : "l"(a.rid_hint + b));
      if (sl >= 4 && sl % 4 == 0 && rid >= 0 && static_cast<uint64_t>(rid) * 8 + 7 < a.state_rows) {
        h_ok = true;
        h_sl = sl;
        h_rid = rid;
        if (line) {
          for (int i = sl == 4 ? 4 : 0; i < 7; ++i) {
            const TIn* row = state + static_cast<size_t>(rid * 8 + (sl - 8 + i) % 8) * width;
            prefetch_l2(row + (i < 4 ? 0 : hd) + c0);
            prefetch_l2(row + (i < 4 ? 2 * hd : 3 * hd) + c0);
          }
        }
      }
    }
  }
  pdl_wait();
  pdl_release();
  float x[VEC] = {0.0f, 0.0f, 0.0f, 0.0f};
  bool stored = false;  // the row goes to the cache (every valid record)
  int64_t pos = 0;
  int64_t loc = -1;
  float4 w = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
  if (live) {
    const ckv_decode_plan_t P = load_plan_d(a.plan_d + b);
    const TIn* src = input + static_cast<size_t>(b) * width + c0;
    const V kv_ovl = ld_stream_v<V>(src), kv_main = ld_stream_v<V>(src + hd);
    const V sc_ovl = ld_stream_v<V>(src + 2 * hd), sc_main = ld_stream_v<V>(src + 3 * hd);
    V ap[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) ap[i] = ld_cached_v<V>(ape + static_cast<size_t>(i) * hd + c0);
    loc = __ldg(n.out_loc + b);
    w = __ldg(reinterpret_cast<const float4*>(n.weight + c0));
    const int h_first = h_sl == 4 ? 4 : 0;
    V kv[8], sc[8];
#pragma unroll
    for (int i = 0; i < 7; ++i) {
      kv[i] = sc[i] = zero_v<V>();
      if (h_ok && i >= h_first) {
        const TIn* row = state + static_cast<size_t>(h_rid * 8 + (h_sl - 8 + i) % 8) * width;
        kv[i] = ld_stream_v<V>(row + (i < 4 ? 0 : hd) + c0);
        sc[i] = ld_stream_v<V>(row + (i < 4 ? 2 * hd : 3 * hd) + c0);
      }
    }
    if (P.seq_len != kInvalidU32) {
      stored = true;
      pos = max(static_cast<int64_t>(P.seq_len) - 4, int64_t{0});
      const bool boundary = P.seq_len % 4 == 0;
      const int64_t rp0 = P.read_page_0, rp1 = P.read_page_1;
      bool ok = P.write_loc >= 0 && static_cast<uint64_t>(P.write_loc) < a.state_rows;
      if (boundary)
        ok = ok && rp0 >= 0 && rp1 >= 0 && static_cast<uint64_t>(rp0) * 4 + 3 < a.state_rows &&
             static_cast<uint64_t>(rp1) * 4 + 3 < a.state_rows;
      if (!ok) {
        if (ch == 0) status_or(a.d_status, CKV_STATUS_BAD_INDEX);
      } else {
        TIn* dst = state + static_cast<size_t>(P.write_loc) * width + c0;
        st_v<V>(dst, kv_ovl);
        st_v<V>(dst + hd, kv_main);
        st_v<V>(dst + 2 * hd, sc_ovl);
        st_v<V>(dst + 3 * hd, sc_main);
        if (boundary) {
          const int first = P.seq_len == 4 ? 4 : 0;
          bool same = h_ok && h_sl == static_cast<int64_t>(P.seq_len);
#pragma unroll
          for (int i = 0; i < 7; ++i)
            if (i >= first) same = same && (i < 4 ? rp0 : rp1) * 4 + (i & 3) == h_rid * 8 + (h_sl - 8 + i) % 8;
          if (!same) {
#pragma unroll
            for (int i = 0; i < 7; ++i) {
              if (i < first) {
                kv[i] = sc[i] = zero_v<V>();
                continue;
              }
              const TIn* row = state + static_cast<size_t>((i < 4 ? rp0 : rp1) * 4 + (i & 3)) * width;
              kv[i] = ld_stream_v<V>(row + (i < 4 ? 0 : hd) + c0);
              sc[i] = ld_stream_v<V>(row + (i < 4 ? 2 * hd : 3 * hd) + c0);
            }
          }
          kv[7] = kv_main;
          sc[7] = sc_main;
          c4_pool_chunk<TIn, VEC>(kv, sc, ap, first, x);
        }
      }
    }
  }
  // RMS of the row: every thread of the block takes part (rows are whole warps)
  float ss = 0.0f;
#pragma unroll
  for (int e = 0; e < VEC; ++e) ss = fmaf(x[e], x[e], ss);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xFFFFFFFFu, ss, off);
  const int warp = threadIdx.x >> 5;
  if ((threadIdx.x & 31) == 0) s_part[warp] = ss;
  __syncthreads();
  const int row_warps = static_cast<int>(chunks) / 32;
  const int w0 = warp / row_warps * row_warps;
  float tot = 0.0f;
  for (int k = 0; k < row_warps; ++k) tot += s_part[w0 + k];
  if (!live || !stored) return;
  const int base = hd - n.rope_dim;
  const bool pos_ok = n.rope_dim == 0 || pos < n.max_pos;
  if (!pos_ok || loc < 0 || static_cast<uint64_t>(loc) >= n.cache_rows) {
    if (ch == 0) status_or(a.d_status, CKV_STATUS_BAD_INDEX);
    return;
  }
  const float r = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(tot, static_cast<float>(hd)), n.eps)));
  float y[4] = {x[0] * r * w.x, x[1] * r * w.y, x[2] * r * w.z, x[3] * r * w.w};
  if (c0 >= base) {  // pairs (c0, c0+1) and (c0+2, c0+3)
    const float4 cs = __ldg(reinterpret_cast<const float4*>(
        n.freqs + (static_cast<size_t>(pos) * (n.rope_dim / 2) + (c0 - base) / 2) * 2));
    const float a0 = y[0], b0 = y[1], a1 = y[2], b1 = y[3];
    y[0] = a0 * cs.x - b0 * cs.y;
    y[1] = a0 * cs.y + b0 * cs.x;
    y[2] = a1 * cs.z - b1 * cs.w;
    y[3] = a1 * cs.w + b1 * cs.z;
  }
  const size_t at = static_cast<size_t>(loc) * hd + c0;
  if (n.cache_dtype == CKV_BF16) {
    *reinterpret_cast<uint2*>(static_cast<uint16_t*>(n.cache) + at) =
        make_uint2(pack_bf16x2(y[0], y[1]), pack_bf16x2(y[2], y[3]));
  } else {
    *reinterpret_cast<float4*>(static_cast<float*>(n.cache) + at) = make_float4(y[0], y[1], y[2], y[3]);
  }
}

// The 4-D view of a [rows, 4 * hd] C4 row tensor, boxes of `box_rows` rows.
int c4_view(CUtensorMap* map, const void* base, int dtype, int hd, uint64_t rows, uint32_t box_rows) {
  const uint64_t esz = dtype == CKV_BF16 ? 2 : 4;
  const uint64_t blk = static_cast<uint64_t>(c4_block(hd));
  const uint64_t q = static_cast<uint64_t>(hd) / blk;
  const uint64_t dims[4] = {blk, 2 * q, 2, rows};
  const uint64_t strides[3] = {blk * esz, 2ull * hd * esz, 4ull * hd * esz};
  const uint32_t box[4] = {static_cast<uint32_t>(blk), static_cast<uint32_t>(q), 2, box_rows};
  return encode_tensor_map(map, dtype, 4, base, dims, strides, box);
}

template <typename TIn, typename TOut, bool kShortWaits, bool kSmall>
int launch_prefill_t(const PoolArgs& a, cudaStream_t s) {
  using S = C4Stage<TIn>;
  const int hd = a.head_dim;
  const uint64_t recs = static_cast<uint64_t>(a.capacity) + (a.out_layout == CKV_OUT_TOKEN ? 1 : 0);
  if (recs == 0) return CKV_OK;
  // tensor-map row coordinates are 32-bit
  if (a.num_q_tokens > 0x7FFFFFFFu || a.state_rows > 0x7FFFFFFFull) return CKV_ERR_SIZE;
  auto fn = c4_pool_prefill_staged_kernel<TIn, TOut, kShortWaits, kSmall>;
  const int R = kSmall ? S::recs_small(hd) : S::recs(hd);
  const int smem = kSmall ? S::stages_small(hd) * static_cast<int>(S::bytes_small(hd))
                          : S::stages(hd) * static_cast<int>(S::bytes(hd));
  const int threads = (R * S::chunks(hd) + 31) / 32 * 32 + 32;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return CKV_ERR_LAUNCH;
  static std::atomic<bool> configured[64];  // per device; a repeated set-up by racing threads is harmless
  if (!configured[dev].load(std::memory_order_acquire)) {
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kC4StageBudget) != cudaSuccess) {
      cudaGetLastError();
      return CKV_ERR_LAUNCH;
    }
    configured[dev].store(true, std::memory_order_release);
  }
  alignas(64) C4Maps maps;
  memset(&maps, 0, sizeof maps);
  int rc = CKV_OK;
  if (a.num_q_tokens > 0) {
    rc = c4_view(&maps.in4, a.input, a.in_dtype, hd, a.num_q_tokens, 4);
    if (!rc) rc = c4_view(&maps.in1, a.input, a.in_dtype, hd, a.num_q_tokens, 1);
  }
  if (!rc && a.state_rows > 0) {
    rc = c4_view(&maps.st4, a.state, a.in_dtype, hd, a.state_rows, 4);
    if (!rc) rc = c4_view(&maps.st1, a.state, a.in_dtype, hd, a.state_rows, 1);
  }
  if (rc) return rc;
  const uint64_t groups = (recs + R - 1) / R;
  const uint64_t per = static_cast<uint64_t>(sm_count()) * (kSmall ? 2 : 1);
  const uint32_t grid = static_cast<uint32_t>(std::max<uint64_t>(1, std::min<uint64_t>(groups, per)));
  return launch_pdl(fn, dim3(grid), dim3(threads), smem, s, a, maps);
}

// Resident blocks per SM of the direct kernel, per device (0: the query
// failed; not cached, so a later launch asks again).
template <typename TIn, typename TOut>
int c4_direct_per_sm() {
  static std::atomic<int> cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  const bool cached_dev = dev >= 0 && dev < 64;
  int per_sm = cached_dev ? cache[dev].load(std::memory_order_relaxed) : 0;
  if (per_sm > 0) return per_sm;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, c4_pool_prefill_direct_kernel<TIn, TOut>,
                                                    kC4DirectThreads, 0) != cudaSuccess ||
      per_sm <= 0) {
    cudaGetLastError();
    return 0;
  }
  if (cached_dev) cache[dev].store(per_sm, std::memory_order_relaxed);
  return per_sm;
}

template <typename TIn, typename TOut>
int launch_prefill_direct_t(const PoolArgs& a, int per_sm, cudaStream_t s) {
  const uint32_t chunks = static_cast<uint32_t>(a.head_dim / C4Vec<TIn>::VEC);
  const uint64_t units64 = (static_cast<uint64_t>(a.capacity) + (a.out_layout == CKV_OUT_TOKEN ? 1 : 0)) * chunks;
  if (units64 == 0) return CKV_OK;
  if (units64 > 0xFFFFFFFFull) return CKV_ERR_SIZE;
  const uint64_t blocks = (units64 + kC4DirectThreads - 1) / kC4DirectThreads;
  const uint32_t grid = static_cast<uint32_t>(
      std::max<uint64_t>(1, std::min<uint64_t>(blocks, static_cast<uint64_t>(per_sm) * sm_count())));
  return launch_pdl(c4_pool_prefill_direct_kernel<TIn, TOut>, dim3(grid), dim3(kC4DirectThreads), 0, s, a, chunks,
                    static_cast<uint32_t>(units64));
}

template <typename TIn, typename TOut>
int launch_decode_t(const PoolArgs& a, cudaStream_t s) {
  const uint32_t chunks = static_cast<uint32_t>(a.head_dim / kC4DecVec);
  const uint64_t units64 = static_cast<uint64_t>(a.capacity) * chunks;
  if (units64 == 0) return CKV_OK;
  if (units64 > 0xFFFFFFFFull) return CKV_ERR_SIZE;
  const uint32_t units = static_cast<uint32_t>(units64);
  // The same number of blocks on every SM: k blocks per SM of at most
  // kC4DecodeMaxThreads threads, k as small as fits, the threads evened out
  // over them.  (A 256-row batch at head_dim 512: 147 blocks of 224 threads
  // against 256 blocks of 128, two on most SMs and one on the rest; in two
  // same-box comparisons the decode step took 8.63-8.75 against 8.73-8.90 us,
  // and back to back 2.64-2.68 against 2.71-2.73 us on one box, the same on
  // the other.)
  const uint64_t sms = static_cast<uint64_t>(sm_count());
  const uint64_t k = (units64 + sms * kC4DecodeMaxThreads - 1) / (sms * kC4DecodeMaxThreads);
  const uint32_t threads = static_cast<uint32_t>(((units64 + k * sms - 1) / (k * sms) + 31) / 32 * 32);
  return launch_pdl(c4_decode_kernel<TIn, TOut>, dim3((units + threads - 1) / threads), dim3(threads), 0, s, a,
                    chunks, units);
}

template <typename TIn>
int launch_decode_norm_t(const PoolArgs& a, const DecodeNormArgs& n, cudaStream_t s) {
  const uint32_t chunks = static_cast<uint32_t>(a.head_dim / kC4DecVec);  // units per row, a multiple of 32
  const uint64_t units64 = static_cast<uint64_t>(a.capacity) * chunks;
  if (units64 == 0) return CKV_OK;
  if (units64 > 0xFFFFFFFFull) return CKV_ERR_SIZE;
  const uint32_t units = static_cast<uint32_t>(units64);
  const uint32_t threads = 128 % chunks == 0 ? 128u : chunks;  // whole rows per block
  return launch_pdl(c4_decode_norm_kernel<TIn>, dim3((units + threads - 1) / threads), dim3(threads), 0, s, a, n,
                    chunks, units);
}

}  // namespace

namespace {

// kernels built for waits shorter than try_wait's window only for such limits
template <typename TIn, typename TOut, bool kSmall>
int launch_prefill_s(const PoolArgs& a, cudaStream_t s) {
  return a.wait_ns < kShortWaitNs ? launch_prefill_t<TIn, TOut, true, kSmall>(a, s)
                                  : launch_prefill_t<TIn, TOut, false, kSmall>(a, s);
}

// Steps of at most eight full stages per SM take the small geometry (two CTAs
// per SM, half the records per stage: 3.34 -> 2.80 us back to back on a
// 16-record step, large steps unchanged), and of those, steps whose records
// fit 1.6 waves of the direct kernel take that one (16 records 2.77 -> 2.29
// us, 1024 records 7.35 -> 6.44 us back to back; at 3.4 waves it took 20.6
// against the staged 17.7 us).  The host knows the plan's capacity, not its
// count, and a padded plan's capacity can be the token count, so the records
// are bounded by the tokens instead: at most ceil(extend / 4) per request of
// a batch of at most 1024, i.e. num_q_tokens / 4 + 768.
template <typename TIn, typename TOut>
int launch_prefill_w(const PoolArgs& a, cudaStream_t s) {
  using S = C4Stage<TIn>;
  const int hd = a.head_dim;
  const bool small = S::recs(hd) >= 2 &&
                     static_cast<uint64_t>(a.capacity) <= static_cast<uint64_t>(8) * sm_count() * S::recs(hd);
  if (!small) return launch_prefill_s<TIn, TOut, false>(a, s);
  const int per_sm = c4_direct_per_sm<TIn, TOut>();
  const uint64_t recs = std::min<uint64_t>(a.capacity, a.num_q_tokens / 4 + 768) +
                        (a.out_layout == CKV_OUT_TOKEN ? 1 : 0);
  const uint64_t units = recs * static_cast<uint64_t>(S::chunks(hd));
  const uint64_t wave = static_cast<uint64_t>(per_sm) * sm_count() * kC4DirectThreads;
  if (per_sm > 0 && units * 5 <= wave * 8) return launch_prefill_direct_t<TIn, TOut>(a, per_sm, s);
  return launch_prefill_s<TIn, TOut, true>(a, s);
}

}  // namespace

int launch_c4_pool_prefill(const PoolArgs& a, cudaStream_t s) {
  if (a.in_dtype == CKV_BF16)
    return a.out_dtype == CKV_BF16 ? launch_prefill_w<__nv_bfloat16, __nv_bfloat16>(a, s)
                                   : launch_prefill_w<__nv_bfloat16, float>(a, s);
  return a.out_dtype == CKV_BF16 ? launch_prefill_w<float, __nv_bfloat16>(a, s) : launch_prefill_w<float, float>(a, s);
}

int launch_c4_decode_norm(const PoolArgs& a, const DecodeNormArgs& n, cudaStream_t s) {
  return a.in_dtype == CKV_BF16 ? launch_decode_norm_t<__nv_bfloat16>(a, n, s) : launch_decode_norm_t<float>(a, n, s);
}

int launch_c4_decode(const PoolArgs& a, cudaStream_t s) {
  if (a.in_dtype == CKV_BF16)
    return a.out_dtype == CKV_BF16 ? launch_decode_t<__nv_bfloat16, __nv_bfloat16>(a, s)
                                   : launch_decode_t<__nv_bfloat16, float>(a, s);
  return a.out_dtype == CKV_BF16 ? launch_decode_t<float, __nv_bfloat16>(a, s) : launch_decode_t<float, float>(a, s);
}

}  // namespace ckv
