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
// Work unit: a tile = (event, slice of CS channels).  The tile's 128 entries x
// CS channels of kv and of score (64 KB) are staged in shared memory by the TMA
// engine and signal one mbarrier, so no register holds staged data.  When all
// 128 entries are consecutive rows of one tensor (a prefill window that lies
// in the extend; the 127 page slots of a decode window) the tile is two 2-D
// tensor-map boxes (kv slice, score slice); a prefill window that starts in the
// state is two row ranges (page slots 0 .. buffer_len-1, then input rows), each
// copied as a few boxes of 64, 16, 4 and 1 rows.  The arithmetic then reads shared
// memory with 8 groups of 16 consecutive entries x CS/4 channel quads: pass 1
// forms the scores and the exact per-channel maximum, pass 2 the group sums of
// weights and weighted kv, pass 3 the fixed pairwise tree over the 8 groups.
// Both kernels below run this same per-thread arithmetic (c128_pass1/2/3), so a
// window gives the same bits whether it is pooled in prefill or in decode.
//
// Both steps run one persistent, warp-specialised kernel: one CTA per SM owns
// one channel slice (its ape slice stays in registers); a producer warp
// streams the CTA's tiles through a shared-memory ring while the consumer
// warps reduce the previous tiles.  Prefill tiles are 128 channels wide (64 KB,
// 3 stages); decode tiles 64 channels (32 KB, 4 stages), and every decode CTA
// first finds the page-boundary rows by a block-wide scan of the plan so that
// the page reads are spread evenly over the SMs.  Decode batches too large for
// that use a kernel with one CTA per (row, slice).
#include <cuda.h>  // CUtensorMap and its enums (types only; the encoder is fetched at run time)

#include <algorithm>
#include <atomic>
#include <cstring>

#include "async_copy.cuh"
#include "common.cuh"
#include "launch.h"

namespace ckv {
namespace {

// A tile of CS channels x 128 entries; 4 channels per thread, 8 entry groups.
template <typename TIn, int CS_>
struct TileCfg {
  static constexpr int CS = CS_;
  static constexpr int QUADS = CS / 4;
  static constexpr int THREADS = QUADS * 8;
  static constexpr int SEG_BYTES = CS * static_cast<int>(sizeof(TIn));  // one entry's kv (or score) slice
  static constexpr int TILE_BYTES = 128 * SEG_BYTES * 2;
  static constexpr int RED_FLOATS = 2 * 8 * CS;                         // group partials (l, a)
};

// Decode: half-width tiles (32 KB) so that several boundary tiles per SM are
// in flight at once.
template <typename TIn>
struct DecodeCfg : TileCfg<TIn, sizeof(TIn) == 2 ? 64 : 32> {
  using Base = TileCfg<TIn, sizeof(TIn) == 2 ? 64 : 32>;
  static constexpr int SMEM = Base::TILE_BYTES + Base::RED_FLOATS * 4;
};

// ---------------------------------------------------------------- tensor-map copies
// (mbarrier and one-dimensional bulk-copy helpers: async_copy.cuh)
// One 2-D tensor-map box (x = column, y = row) -> shared memory.
__device__ __forceinline__ void tma_box_g2s(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

// One 2-D tensor-map box into L2 only (no shared memory, no barrier).
__device__ __forceinline__ void tma_box_prefetch_l2(const CUtensorMap* map, int x, int y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y)
               : "memory");
}

__device__ __forceinline__ void prefetch_map(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ---------------------------------------------------------------- element helpers
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

// Zero rows [r0, r1) of out, columns [c0, c0 + CS), with NT threads.
template <int CS, typename TOut, int NT>
__device__ __forceinline__ void zero_rows(TOut* out, int hd, int c0, int64_t r0, int64_t r1, int t) {
  constexpr int kPerRow = CS * static_cast<int>(sizeof(TOut)) / 16;
  constexpr int kElems = 16 / static_cast<int>(sizeof(TOut));
  const int64_t total = (r1 - r0) * kPerRow;
  for (int64_t idx = t; idx < total; idx += NT) {
    const int64_t r = r0 + idx / kPerRow;
    const int c = c0 + static_cast<int>(idx % kPerRow) * kElems;
    st16(out + r * hd + c, make_uint4(0, 0, 0, 0));
  }
}

// ---------------------------------------------------------------- the per-thread arithmetic
// Thread (q, g) owns channels cq = 4q .. 4q+3 of the tile (two fp32 pairs) and
// entries 16g .. 16g+15.  ape_at(k, v) yields ape[16g + k][c0 + cq + 0..3] as
// two fp32 pairs.

// Four channels of a staged entry as two fp32 pairs.
template <typename TIn>
__device__ __forceinline__ void load4x2(const TIn* p, F2 (&v)[2]);

template <>
__device__ __forceinline__ void load4x2<__nv_bfloat16>(const __nv_bfloat16* p, F2 (&v)[2]) {
  const uint2 u = *reinterpret_cast<const uint2*>(p);
  v[0] = f2_from_bf16x2(u.x);
  v[1] = f2_from_bf16x2(u.y);
}

template <>
__device__ __forceinline__ void load4x2<float>(const float* p, F2 (&v)[2]) {
  const float4 u = *reinterpret_cast<const float4*>(p);
  v[0] = f2_pack(u.x, u.y);
  v[1] = f2_pack(u.z, u.w);
}

// The same from global memory through the read-only path (ape).
template <typename TIn>
__device__ __forceinline__ void ldg4x2(const TIn* p, F2 (&v)[2]) {
  float f[4];
  ldg4<TIn>(p, f);
  v[0] = f2_pack(f[0], f[1]);
  v[1] = f2_pack(f[2], f[3]);
}

__device__ __forceinline__ void max_into(float (&m)[4], const F2 (&s)[2]) {
  float x0, x1, x2, x3;
  f2_unpack(s[0], x0, x1);
  f2_unpack(s[1], x2, x3);
  m[0] = fmaxf(m[0], x0);
  m[1] = fmaxf(m[1], x1);
  m[2] = fmaxf(m[2], x2);
  m[3] = fmaxf(m[3], x3);
}

template <typename TIn, int CS, typename ApeAt>
__device__ __forceinline__ void c128_pass1(const TIn* sc_s, int g, int cq, ApeAt ape_at, F2 (&s)[16][2],
                                           float (&m)[4]) {
#pragma unroll
  for (int j = 0; j < 4; ++j) m[j] = -INFINITY;
#pragma unroll
  for (int k = 0; k < 16; ++k) {
    F2 sc[2], bias[2];
    load4x2<TIn>(sc_s + (16 * g + k) * CS + cq, sc);
    ape_at(k, bias);
    s[k][0] = score_plus_bias2(sc[0], bias[0]);
    s[k][1] = score_plus_bias2(sc[1], bias[1]);
    max_into(m, s[k]);
  }
}

template <typename TIn, int CS>
__device__ __forceinline__ void c128_pass2(const TIn* kv_s, int g, int cq, const F2 (&s)[16][2], const F2 (&nml)[2],
                                           PoolAcc2 (&acc)[2]) {
  acc[0].init();
  acc[1].init();
#pragma unroll
  for (int k = 0; k < 16; ++k) {
    F2 kv[2];
    load4x2<TIn>(kv_s + (16 * g + k) * CS + cq, kv);
    acc[0].add(kv[0], weight_of2(s[k][0], nml[0]));
    acc[1].add(kv[1], weight_of2(s[k][1], nml[1]));
  }
}

// The same pass 2 without cached scores: s is formed again from the staged
// score and ape with the same single rounding, so the result is identical.
template <typename TIn, int CS, typename ApeAt>
__device__ __forceinline__ void c128_pass2_recompute(const TIn* kv_s, const TIn* sc_s, int g, int cq, ApeAt ape_at,
                                                     const F2 (&nml)[2], PoolAcc2 (&acc)[2]) {
  acc[0].init();
  acc[1].init();
#pragma unroll
  for (int k = 0; k < 16; ++k) {
    F2 kv[2], sc[2], bias[2];
    load4x2<TIn>(kv_s + (16 * g + k) * CS + cq, kv);
    load4x2<TIn>(sc_s + (16 * g + k) * CS + cq, sc);
    ape_at(k, bias);
    acc[0].add(kv[0], weight_of2(score_plus_bias2(sc[0], bias[0]), nml[0]));
    acc[1].add(kv[1], weight_of2(score_plus_bias2(sc[1], bias[1]), nml[1]));
  }
}

// Pass 1 without keeping the scores: only the per-channel maximum.
template <typename TIn, int CS, typename ApeAt>
__device__ __forceinline__ void c128_max_only(const TIn* sc_s, int g, int cq, ApeAt ape_at, float (&m)[4]) {
#pragma unroll
  for (int j = 0; j < 4; ++j) m[j] = -INFINITY;
#pragma unroll
  for (int k = 0; k < 16; ++k) {
    F2 sc[2], bias[2], s[2];
    load4x2<TIn>(sc_s + (16 * g + k) * CS + cq, sc);
    ape_at(k, bias);
    s[0] = score_plus_bias2(sc[0], bias[0]);
    s[1] = score_plus_bias2(sc[1], bias[1]);
    max_into(m, s);
  }
}

// Channel maximum over the 8 groups' partial maxima (exact in any order),
// returned as -max*log2(e) for the channel pairs.
template <int CS>
__device__ __forceinline__ void c128_nml(const float* red_m, int cq, F2 (&nml)[2]) {
  float n[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    float mm = red_m[cq + j];
#pragma unroll
    for (int gg = 1; gg < 8; ++gg) mm = fmaxf(mm, red_m[gg * CS + cq + j]);
    n[j] = neg_max_log2e(mm);
  }
  nml[0] = f2_pack(n[0], n[1]);
  nml[1] = f2_pack(n[2], n[3]);
}

// Group partials (l, a) of the four channels into the reduction buffers.
template <int CS>
__device__ __forceinline__ void store_partials(float* red_l, float* red_a, int g, int cq, const PoolAcc2 (&acc)[2]) {
  float l0, l1, l2, l3, a0, a1, a2, a3;
  f2_unpack(acc[0].l, l0, l1);
  f2_unpack(acc[1].l, l2, l3);
  f2_unpack(acc[0].a, a0, a1);
  f2_unpack(acc[1].a, a2, a3);
  *reinterpret_cast<float4*>(red_l + g * CS + cq) = make_float4(l0, l1, l2, l3);
  *reinterpret_cast<float4*>(red_a + g * CS + cq) = make_float4(a0, a1, a2, a3);
}

template <typename TIn>
__device__ __forceinline__ void load_ape_regs(const TIn* ape, int hd, int c0, int g, int cq, F2 (&ape_r)[16][2]) {
#pragma unroll
  for (int k = 0; k < 16; ++k) ldg4x2<TIn>(ape + static_cast<size_t>(16 * g + k) * hd + c0 + cq, ape_r[k]);
}

// Tensor maps for prefill windows that start in the state: the state and the
// input, each with boxes of gather_height(k) rows x one channel slice.  A
// row range of n < 128 rows then takes at most 10 boxes (64, 16 x 3, 4 x 3,
// 1 x 3) per half: the copy engine handles a handful of operations per tile
// instead of one per row.
__host__ __device__ constexpr int gather_height(int k) { return 64 >> (2 * k); }  // 64, 16, 4, 1

struct GatherMaps {
  CUtensorMap state[4];
  CUtensorMap input[4];
};

// Issues the copies of one prefill tile whose window starts in the state (one
// thread): entries 0 .. bl-1 are page rows y_state .. y_state+bl-1, entries
// bl .. 127 input rows y_input .. y_input+127-bl.
template <typename TIn, int CS>
__device__ __forceinline__ void issue_gather(TIn* kv_s, const GatherMaps& gm, int hd, int c0, int y_state,
                                             int y_input, int bl, uint32_t bar) {
  TIn* sc_s = kv_s + 128 * CS;
  int e = 0;
  auto range = [&](const CUtensorMap* maps, int y, int n) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int h = gather_height(k);
      while (n >= h) {
        tma_box_g2s(smem_addr(kv_s + e * CS), &maps[k], c0, y, bar);
        tma_box_g2s(smem_addr(sc_s + e * CS), &maps[k], hd + c0, y, bar);
        e += h;
        y += h;
        n -= h;
      }
    }
  };
  range(gm.state, y_state, bl);
  range(gm.input, y_input, 128 - bl);
}

// Issues decode tile n's copies into stage buffer kv_s: page slots 0..126 as
// two 127-row boxes, entry 127 = the new token's input row (one thread).
template <typename TIn, int CS>
__device__ __forceinline__ void issue_decode_tile(TIn* kv_s, uint32_t bar, const CUtensorMap* page_map,
                                                  const TIn* input, size_t width, int hd, int c0, uint32_t row,
                                                  int32_t page) {
  using T = TileCfg<TIn, CS>;
  mbar_arrive_expect_tx(bar, T::TILE_BYTES);
  const int y = static_cast<int>(static_cast<int64_t>(page) * 128);
  tma_box_g2s(smem_addr(kv_s), page_map, c0, y, bar);
  tma_box_g2s(smem_addr(kv_s + 128 * CS), page_map, hd + c0, y, bar);
  const TIn* in_row = input + static_cast<size_t>(row) * width;
  bulk_g2s(smem_addr(kv_s + 127 * CS), in_row + c0, T::SEG_BYTES, bar);
  bulk_g2s(smem_addr(kv_s + 128 * CS + 127 * CS), in_row + hd + c0, T::SEG_BYTES, bar);
}

// Decodes and bounds-checks prefill record e.  Invalid (padding) records and
// records that point outside the state / input return false.
__device__ __forceinline__ bool prefill_record_of(const PoolArgs& a, const ckv_compress_plan_t& P, uint32_t& ragged,
                                                  int& bl, int64_t& rp0, bool& bad) {
  bad = false;
  if (plan_c_invalid(P)) return false;
  ragged = P.ragged_bl & CKV_RAGGED_MASK;
  bl = static_cast<int>(P.ragged_bl >> CKV_BUFFER_LEN_SHIFT);
  rp0 = P.read_page_0;
  bool ok = ragged < a.num_q_tokens && bl <= 127 && static_cast<int64_t>(ragged) - 127 + bl >= 0;
  if (bl > 0) ok = ok && rp0 >= 0 && static_cast<uint64_t>(rp0) * 128 + 127 < a.state_rows;
  bad = !ok;
  return ok;
}

__device__ __forceinline__ bool prefill_record(const PoolArgs& a, uint32_t e, uint32_t& ragged, int& bl,
                                               int64_t& rp0, bool& bad) {
  return prefill_record_of(a, load_plan_c(a.plan_c + e), ragged, bl, rp0, bad);
}

// Record e of the plan buffer, or the invalid record past its capacity.  A
// record inside the buffer may be read before the count is known.
__device__ __forceinline__ ckv_compress_plan_t plan_c_at(const PoolArgs& a, uint32_t e) {
  if (e < a.capacity) return load_plan_c(a.plan_c + e);
  ckv_compress_plan_t P;
  P.seq_len = kInvalidU32;
  P.ragged_bl = kInvalidU32;
  P.read_page_0 = P.read_page_1 = -1;
  return P;
}

// ---------------------------------------------------------------- persistent kernel
// One CTA per SM, bound to one channel slice; its ape slice stays in
// registers.  A producer warp streams the CTA's tiles through an NS-stage ring
// of shared-memory tiles; the consumer warps reduce them.
//   prefill: the CTA's tiles are compress records first, first + per_slice, ...
//   decode:  every CTA first block-scans the decode plan for page-boundary rows
//            and keeps the ones of rank first, first + per_slice, ...; it also
//            does the state write / zero output of rows blockIdx, blockIdx +
//            gridDim, ... (the part of decode that reads no page).
constexpr int kOwnRows = 512;   // decode: rows one CTA may own (boundary rows; rows it writes)
// decode: tiles a producer keeps in flight (measured back to back on 512 rows
// with the boundary-row list: lag 2 / 3 -> 9.23 / 9.09 us with 4 stages,
// 9.25 / 9.10 us with 6)
constexpr int kDecLag = 3;
// decode: plan rows each thread examines per scan pass (measured with the
// paced producer: 1 / 2 / 3 / 4 rows -> 10.17 / 9.22 / 9.56 / 9.85 us back to
// back on 512 rows)
constexpr int kScanK = 2;

template <typename TIn, int CS, int NS, int NG, bool kDecode>
struct PersistCfg {
  using T = TileCfg<TIn, CS>;
  static constexpr int NCG = T::THREADS;   // threads of one consumer group
  static constexpr int NC = NG * NCG;      // all consumer threads
  static constexpr int NSIDE = kDecode ? 64 : 0;  // decode: side warps for the rows that read no page
  static constexpr int THREADS = NC + 32 + NSIDE;  // + the producer warp
  static constexpr int SMEM = NS * T::TILE_BYTES + 2 * NG * T::RED_FLOATS * 4 + (kDecode ? kOwnRows * 24 : 0);
  static_assert(NS % NG == 0, "each consumer group owns every NG-th stage");
};

// Decode plan row r: valid (in range) and on a page boundary?  One coherent
// 16-byte load that the compiler may not repeat later (a read-only load could
// be re-issued after the scan's barriers, a second memory round trip).
__device__ __forceinline__ bool decode_row(const PoolArgs& a, uint32_t r, bool& valid, bool& boundary,
                                           ckv_decode_plan_t& P) {
  uint4 v;
  asm volatile("ld.global.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(a.plan_d + r));
  P.seq_len = v.x;
  P.write_loc = static_cast<int32_t>(v.y);
  P.read_page_0 = static_cast<int32_t>(v.z);
  P.read_page_1 = static_cast<int32_t>(v.w);
  valid = false;
  boundary = false;
  if (P.seq_len == kInvalidU32) return false;  // invalid record: zero output, nothing else
  boundary = P.seq_len % 128 == 0;
  valid = P.write_loc >= 0 && static_cast<uint64_t>(P.write_loc) < a.state_rows;
  if (boundary)
    valid = valid && P.read_page_0 >= 0 && static_cast<uint64_t>(P.read_page_0) * 128 + 127 < a.state_rows;
  return true;
}

// Entry of the boundary list (ckv_decode_order_t, written by the previous
// kernel: a coherent load).  Entries that point outside the batch or the
// state come back as {kInvalidU32, 0}.
__device__ __forceinline__ uint2 load_order_entry(const PoolArgs& a, uint32_t idx) {
  uint2 v;
  asm volatile("ld.global.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(a.order + idx));
  const int32_t page = static_cast<int32_t>(v.y);
  const bool ok = v.x < a.capacity && page >= 0 && static_cast<uint64_t>(page) * 128 + 127 < a.state_rows;
  return ok ? v : make_uint2(kInvalidU32, 0u);
}

__device__ __forceinline__ uint32_t load_order_count(const PoolArgs& a) {
  uint32_t v;
  asm volatile("ld.global.u32 %0, [%1];" : "=r"(v) : "l"(a.order));
  return v;
}

// The rows of a decode step that read no page: every row in `rows` ({row,
// write_loc, flags}) writes its new token to its slot (never one of the 127
// slots any window reads), and rows that emit nothing get a zero output row.
constexpr uint32_t kRowValid = 1u, kRowBoundary = 2u;

// They are written by the side warps (NTH threads), which do nothing else: a
// batch of rows has all its input chunks in flight before the first store.
template <typename TIn, typename TOut, int NTH>
__device__ __forceinline__ void decode_rows_side(const PoolArgs& a, const uint4* rows, uint32_t nrows, int tl) {
  constexpr int kVec = 16 / static_cast<int>(sizeof(TIn));
  constexpr int kOutVec = 16 / static_cast<int>(sizeof(TOut));
  constexpr int kRows = 4;    // rows per batch
  constexpr int kChunks = 4;  // 16-byte chunks per thread and row per round
  const int hd = a.head_dim;
  const int width = 2 * hd;
  const int in_chunks = width / kVec;
  const int out_chunks = hd / kOutVec;
  const TIn* input = static_cast<const TIn*>(a.input);
  TIn* state = static_cast<TIn*>(a.state_mut);
  TOut* out = static_cast<TOut*>(a.out);
  for (uint32_t base = 0; base < nrows; base += kRows) {
    uint4 rec[kRows];
#pragma unroll
    for (int k = 0; k < kRows; ++k) rec[k] = base + k < nrows ? rows[base + k] : make_uint4(0, 0, 0, 0);
    for (int cb = 0; cb < in_chunks; cb += kChunks * NTH) {
      uint4 v[kRows][kChunks];
#pragma unroll
      for (int k = 0; k < kRows; ++k)
#pragma unroll
        for (int j = 0; j < kChunks; ++j) {
          const int c = cb + j * NTH + tl;
          if (c < in_chunks && (rec[k].z & kRowValid))
            v[k][j] = ld_stream16(input + static_cast<size_t>(rec[k].x) * width + c * kVec);
        }
#pragma unroll
      for (int k = 0; k < kRows; ++k)
#pragma unroll
        for (int j = 0; j < kChunks; ++j) {
          const int c = cb + j * NTH + tl;
          if (c < in_chunks && (rec[k].z & kRowValid))
            st16(state + static_cast<size_t>(rec[k].y) * width + c * kVec, v[k][j]);
        }
    }
#pragma unroll
    for (int k = 0; k < kRows; ++k) {
      if (base + k < nrows && !((rec[k].z & kRowValid) && (rec[k].z & kRowBoundary)))
        for (int c = tl; c < out_chunks; c += NTH)
          st16(out + static_cast<size_t>(rec[k].x) * hd + c * kOutVec, make_uint4(0, 0, 0, 0));
    }
  }
}

__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

// The ape slice into registers with loads the compiler keeps where they are
// written (issued at once, used by the first tile).
template <typename TIn>
__device__ __forceinline__ void load_ape_regs_now(const TIn* ape, int hd, int c0, int g, int cq, F2 (&ape_r)[16][2]) {
#pragma unroll
  for (int k = 0; k < 16; ++k) {
    const TIn* p = ape + static_cast<size_t>(16 * g + k) * hd + c0 + cq;
    if constexpr (sizeof(TIn) == 2) {
      uint32_t x, y;
      asm volatile("ld.global.nc.v2.u32 {%0, %1}, [%2];" : "=r"(x), "=r"(y) : "l"(p));
      ape_r[k][0] = f2_from_bf16x2(x);
      ape_r[k][1] = f2_from_bf16x2(y);
    } else {
      float x, y, z, w;
      asm volatile("ld.global.nc.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(x), "=f"(y), "=f"(z), "=f"(w) : "l"(p));
      ape_r[k][0] = f2_pack(x, y);
      ape_r[k][1] = f2_pack(z, w);
    }
  }
}

// Consumer barrier of group `grp` (ids 1 .. NG), N threads.
__device__ __forceinline__ void group_sync(int grp, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(1 + grp), "r"(n) : "memory");
}

__device__ __forceinline__ bool group_any(int grp, int n, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(pred)), "r"(1 + grp), "r"(n)
      : "memory");
  return r != 0;
}

template <typename TIn, typename TOut, int CS, int NS, int NG, bool kDecode, bool kShortWaits>
__global__ __launch_bounds__(PersistCfg<TIn, CS, NS, NG, kDecode>::THREADS, 1) void c128_persistent_kernel(
    const PoolArgs a, uint32_t slices, const __grid_constant__ CUtensorMap in_map,
    const __grid_constant__ CUtensorMap page_map, const __grid_constant__ GatherMaps gather) {
  using T = TileCfg<TIn, CS>;
  using Cfg = PersistCfg<TIn, CS, NS, NG, kDecode>;
  constexpr int NCG = Cfg::NCG;
  constexpr int NC = Cfg::NC;
  constexpr int NT = Cfg::THREADS;
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t full_bar[NS];
  __shared__ __align__(8) uint64_t empty_bar[NS];
  __shared__ volatile int abort_flag;
  __shared__ uint32_t s_warp_count[NT / 32];
  float* red_base = reinterpret_cast<float*>(smem + NS * T::TILE_BYTES);
  uint4* trivrow = reinterpret_cast<uint4*>(smem + NS * T::TILE_BYTES + 2 * NG * T::RED_FLOATS * 4);
  uint2* own = reinterpret_cast<uint2*>(trivrow + kOwnRows);

  const int t = threadIdx.x;
  const int warp = t >> 5;
  const int lane = t & 31;
  const uint32_t slice = blockIdx.x % slices;
  const uint32_t first = blockIdx.x / slices;
  const uint32_t stride = gridDim.x / slices;
  const int c0 = static_cast<int>(slice) * CS;
  const int hd = a.head_dim;
  const size_t width = 2 * static_cast<size_t>(hd);
  const TIn* input = static_cast<const TIn*>(a.input);
  const TIn* state = kDecode ? static_cast<const TIn*>(a.state_mut) : static_cast<const TIn*>(a.state);
  TOut* out = static_cast<TOut*>(a.out);
  const bool token = !kDecode && a.out_layout == CKV_OUT_TOKEN;

  if (t == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(smem_addr(&full_bar[s]), 1);
      mbar_init(smem_addr(&empty_bar[s]), NCG / 32);
    }
    abort_flag = 0;
    fence_mbar_init();
  }
  const int grp = t / NCG;
  const int tl = t % NCG;
  const int q = tl % T::QUADS;
  const int g = tl / T::QUADS;
  const int cq = 4 * q;
  F2 ape_r[16][2];
  // the tensor map is a kernel parameter: fetch its descriptor while the plan is scanned
  if (warp == NC / 32) {
    if (lane == 0) prefetch_map(kDecode ? &page_map : &in_map);
    if (!kDecode && lane >= 1 && lane <= 8)
      prefetch_map(lane <= 4 ? &gather.state[lane - 1] : &gather.input[lane - 5]);
  }

  const bool ordered = kDecode && a.order != nullptr;
  if (ordered) {
    // Warm the L2 (and the address translations) for this CTA's first loads
    // while the previous kernel finishes: its list entries, the records and
    // input rows of the rows it writes, its ape slice.  L2 is coherent, so
    // lines the previous kernel still writes are read correctly after the wait.
    const uint32_t B = a.capacity;
    const uint32_t cap = B > first ? (B - first + stride - 1) / stride : 0u;
    const uint32_t nt = B > blockIdx.x ? (B - blockIdx.x + gridDim.x - 1) / gridDim.x : 0u;
    if (t == 0) prefetch_l2(a.order);
    if (static_cast<uint32_t>(t) < cap) prefetch_l2(a.order + 1 + first + t * stride);
    if (static_cast<uint32_t>(t) < nt) prefetch_l2(a.plan_d + blockIdx.x + t * gridDim.x);
    if (t < 128) prefetch_l2(static_cast<const TIn*>(a.ape) + static_cast<size_t>(t) * hd + c0);
    const int lines = static_cast<int>(width * sizeof(TIn) / 128);  // of one input row
    for (int i = t; i < static_cast<int>(nt) * lines; i += NT)
      prefetch_l2(reinterpret_cast<const uint8_t*>(input) + (blockIdx.x + (i / lines) * static_cast<size_t>(gridDim.x)) *
                                                                 width * sizeof(TIn) + (i % lines) * 128);
  }
  if (kDecode && a.seq_hint != nullptr) {
    // Windows into L2 while the previous kernel drains: the rows this CTA
    // writes (blockIdx, blockIdx + gridDim, ...) that end a page get their
    // 127 page slots prefetched, every channel slice (whichever CTA pools
    // them then finds them in L2).  The hints are read before the dependency
    // wait, so they only steer prefetches: a stale value costs bandwidth,
    // never a result; pages outside the state are not touched.
    const uint32_t B = a.capacity;
    const uint32_t nt = B > blockIdx.x ? (B - blockIdx.x + gridDim.x - 1) / gridDim.x : 0u;
    for (uint32_t k = t; k < nt; k += NT) {
      const uint32_t r = blockIdx.x + k * gridDim.x;
      int64_t sl, rid;
      asm volatile("ld.global.u64 %0, [%1];" : "=l"(sl) : "l"(a.seq_hint + r));
      asm volatile("ld.global.u64 %0, [%1];" : "=l"(rid) : "l"(a.rid_hint + r));
      if (sl >= 128 && sl % 128 == 0 && rid >= 0 && rid < 0x7FFFFFFF / 128 &&
          static_cast<uint64_t>(rid) * 128 + 127 < a.state_rows) {
        const int y = static_cast<int>(rid * 128);
        for (int x = 0; x < 2 * hd; x += CS) tma_box_prefetch_l2(&page_map, x, y);
      }
    }
  }
  if (!kDecode && a.ext_hint != nullptr) {
    // Prefill (small steps only, see the host): the windows that start in the
    // state -- a request's first window when its prefix ends inside a page --
    // into L2 while the planner runs: page rows rid*128 .. rid*128 + pl%128 - 1,
    // contiguous, for every channel slice.  One thread per request; the hints
    // are the planner's own inputs, read before the dependency wait, so they
    // only steer prefetches.
    for (uint32_t b = blockIdx.x + static_cast<uint32_t>(t) * gridDim.x; b < a.hint_batch;
         b += static_cast<uint32_t>(NT) * gridDim.x) {
      int64_t sl, el, rid;
      asm volatile("ld.global.u64 %0, [%1];" : "=l"(sl) : "l"(a.seq_hint + b));
      asm volatile("ld.global.u64 %0, [%1];" : "=l"(el) : "l"(a.ext_hint + b));
      asm volatile("ld.global.u64 %0, [%1];" : "=l"(rid) : "l"(a.rid_hint + b));
      const int64_t pl = sl - el;
      if (el > 0 && pl > 0 && sl / 128 > pl / 128 && pl % 128 != 0 && rid >= 0 &&
          rid < (int64_t{1} << 48) && static_cast<uint64_t>(rid) * 128 + 127 < a.state_rows) {
        const uint8_t* p = reinterpret_cast<const uint8_t*>(state + static_cast<size_t>(rid) * 128 * width);
        const uint32_t bytes = static_cast<uint32_t>(pl % 128) * static_cast<uint32_t>(width * sizeof(TIn));
        for (uint32_t o = 0; o < bytes; o += 32768u) bulk_prefetch_l2(p + o, bytes - o < 32768u ? bytes - o : 32768u);
      }
    }
  }
  pdl_wait();  // everything below may read what the previous kernel wrote
  pdl_release();
  if (ordered && t < NC) load_ape_regs_now<TIn>(static_cast<const TIn*>(a.ape), hd, c0, g, cq, ape_r);
  // prefill: the producer requests its first record together with the count
  // instead of after it (one dependent round trip less before the first tile)
  ckv_compress_plan_t rec_next = plan_c_at(a, !kDecode && t == NC ? first : kInvalidU32);
  const uint32_t num_c = kDecode ? 0u : count_or_capacity(a.d_counts, 0, a.capacity);
  uint32_t items, ntriv = 0;
  __shared__ uint32_t s_count;
  if (ordered) {
    // The boundary list gives this CTA its windows directly: entries of rank
    // first, first + stride, ... ({row, page}), loaded together with the
    // records of the rows it writes (rows blockIdx, blockIdx + gridDim, ...)
    // in one round of loads.  Thread 0 also loads the count and issues the
    // first tile as soon as its entry is in (stage 0 is free; the producer
    // starts at the second).  The host keeps both shares below kOwnRows.
    const uint32_t B = a.capacity;
    const uint32_t cap = B > first ? (B - first + stride - 1) / stride : 0u;
    ntriv = B > blockIdx.x ? (B - blockIdx.x + gridDim.x - 1) / gridDim.x : 0u;
    const uint32_t count = t == 0 ? load_order_count(a) : 0u;
    const uint32_t nk = cap > ntriv ? cap : ntriv;
    for (uint32_t k = t; k < nk; k += NT) {
      uint2 e = make_uint2(kInvalidU32, 0u);
      if (k < cap) e = load_order_entry(a, 1 + first + k * stride);
      if (k < ntriv) {
        const uint32_t r = blockIdx.x + k * gridDim.x;
        bool valid = false, boundary = false;
        ckv_decode_plan_t P;
        const bool rec = decode_row(a, r, valid, boundary, P);
        trivrow[k] = make_uint4(r, static_cast<uint32_t>(P.write_loc),
                                (valid ? kRowValid : 0u) | (boundary ? kRowBoundary : 0u), 0u);
        if (rec && !valid) status_or(a.d_status, CKV_STATUS_BAD_INDEX);
      }
      if (k < cap) own[k] = e;
      if (k == 0 && cap > 0 && first < count) {
        if (e.x != kInvalidU32) {
          issue_decode_tile<TIn, CS>(reinterpret_cast<TIn*>(smem), smem_addr(&full_bar[0]), &page_map, input, width,
                                     hd, c0, e.x, static_cast<int32_t>(e.y));
        } else {
          status_or(a.d_status, CKV_STATUS_BAD_INDEX);
          mbar_arrive_expect_tx(smem_addr(&full_bar[0]), 0u);
        }
      }
    }
    if (t == 0) s_count = count;
    __syncthreads();
    const uint32_t total = s_count;
    items = total > first ? (total - first + stride - 1) / stride : 0u;
    if (items > cap) items = cap;
  } else if constexpr (kDecode) {
    // Ranks of the page-boundary rows (in row order) by block-wide scans: in
    // each pass thread t looks at kScanK consecutive rows.  This CTA owns the
    // boundary rows of rank first, first + stride, ... ({row, page} pairs) and
    // writes the state / zero rows of rows blockIdx, blockIdx + gridDim, ...
    // (the host keeps both counts below kOwnRows).
    const uint32_t B = a.capacity;
    uint32_t seen = 0;
    for (uint32_t base = 0; base < B; base += kScanK * NT) {
      bool take[kScanK];
      ckv_decode_plan_t P[kScanK];
      uint32_t cnt = 0;
#pragma unroll
      for (int k = 0; k < kScanK; ++k) {
        const uint32_t r = base + t * kScanK + k;
        bool valid = false, boundary = false;
        if (r < B) {
          const bool rec = decode_row(a, r, valid, boundary, P[k]);
          if (r % gridDim.x == blockIdx.x) {
            trivrow[r / gridDim.x] = make_uint4(r, static_cast<uint32_t>(P[k].write_loc),
                                                (valid ? kRowValid : 0u) | (boundary ? kRowBoundary : 0u), 0u);
            if (rec && !valid) status_or(a.d_status, CKV_STATUS_BAD_INDEX);
          }
        }
        take[k] = r < B && valid && boundary;
        cnt += take[k] ? 1u : 0u;
      }
      uint32_t incl = cnt;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const uint32_t v = __shfl_up_sync(0xFFFFFFFFu, incl, off);
        if (lane >= off) incl += v;
      }
      if (lane == 31) s_warp_count[warp] = incl;
      __syncthreads();
      uint32_t rank = seen + incl - cnt, total = seen;
#pragma unroll
      for (int w = 0; w < NT / 32; ++w) {
        const uint32_t c = s_warp_count[w];
        if (w < warp) rank += c;
        total += c;
      }
#pragma unroll
      for (int k = 0; k < kScanK; ++k) {
        if (take[k]) {
          if (rank % stride == first) {
            const uint32_t r = base + t * kScanK + k;
            own[rank / stride] = make_uint2(r, static_cast<uint32_t>(P[k].read_page_0));
            // the thread that finds this CTA's first tile issues it at once
            // (stage 0 is free); the producer starts at the second
            if (rank == first)
              issue_decode_tile<TIn, CS>(reinterpret_cast<TIn*>(smem), smem_addr(&full_bar[0]), &page_map, input,
                                         width, hd, c0, r, P[k].read_page_0);
          }
          ++rank;
        }
      }
      seen = total;
      __syncthreads();
    }
    items = seen > first ? (seen - first + stride - 1) / stride : 0u;
    ntriv = B > blockIdx.x ? (B - blockIdx.x + gridDim.x - 1) / gridDim.x : 0u;
  } else {
    __syncthreads();
    items = num_c > first ? (num_c - first + stride - 1) / stride : 0u;
  }

  if constexpr (kDecode) {
    if (t >= NC + 32) {  // ---------------- side warps: the rows that read no page
      decode_rows_side<TIn, TOut, Cfg::NSIDE>(a, trivrow, ntriv, t - (NC + 32));
      return;
    }
  }
  if (warp == NC / 32) {
    // ---------------- producer: lane 0 of the producer warp alone issues every
    // copy and takes every wait (decode: tile 0 was issued by the scan)
    if (lane != 0) return;
    uint32_t n = kDecode && items > 0 ? 1u : 0u;  // tiles issued so far
    for (; n < items; ++n) {
      const int stage = static_cast<int>(n % NS);
      const uint32_t phase = (n / NS) & 1u;
      // decode: at most kDecLag tiles in flight (tile n >= kDecLag waits for
      // tile n - kDecLag to land).  Every SM asking for its whole ring at once
      // made each first tile wait for the whole burst; pacing the issue lets
      // the first tiles land, and the reductions start, earlier.  (kDecLag <
      // NS: that tile's stage is not refilled before tile n is issued, so its
      // phase is exact.)
      if ((kDecode && n >= static_cast<uint32_t>(kDecLag) &&
           !wait_for<kShortWaits>(smem_addr(&full_bar[(n - kDecLag) % NS]), ((n - kDecLag) / NS) & 1u,
                                  a.wait_ns)) ||
          !wait_for<kShortWaits>(smem_addr(&empty_bar[stage]), phase ^ 1u, a.wait_ns)) {
        status_or(a.d_status, CKV_STATUS_TIMEOUT);
        abort_flag = 1;
        break;
      }
      if (abort_flag) break;  // a consumer gave up: issue nothing more
      const uint32_t bar = smem_addr(&full_bar[stage]);
      TIn* kv_s = reinterpret_cast<TIn*>(smem + stage * T::TILE_BYTES);
      if constexpr (kDecode) {
        const uint2 rp = own[n];
        if (rp.x != kInvalidU32) {
          issue_decode_tile<TIn, CS>(kv_s, bar, &page_map, input, width, hd, c0, rp.x, static_cast<int32_t>(rp.y));
        } else {  // a list entry outside the batch or the state
          status_or(a.d_status, CKV_STATUS_BAD_INDEX);
          mbar_arrive_expect_tx(bar, 0u);
        }
      } else {
        // each record is requested one tile ahead
        const ckv_compress_plan_t P = rec_next;
        if (n + 1 < items) rec_next = plan_c_at(a, first + (n + 1) * stride);
        uint32_t ragged = 0;
        int bl = 0;
        int64_t rp0 = 0;
        bool bad;
        const bool ok = prefill_record_of(a, P, ragged, bl, rp0, bad);
        if (bad) status_or(a.d_status, CKV_STATUS_BAD_INDEX);
        mbar_arrive_expect_tx(bar, ok ? T::TILE_BYTES : 0u);
        if (ok) {
          if (bl == 0) {  // rows ragged-127 .. ragged of the input: two boxes
            tma_box_g2s(smem_addr(kv_s), &in_map, c0, static_cast<int>(ragged) - 127, bar);
            tma_box_g2s(smem_addr(kv_s + 128 * CS), &in_map, hd + c0, static_cast<int>(ragged) - 127, bar);
          } else {
            issue_gather<TIn, CS>(kv_s, gather, hd, c0, static_cast<int>(rp0 * 128),
                                  static_cast<int>(ragged) - 127 + bl, bl, bar);
          }
        }
      }
    }
    // the last NS tiles issued (one per stage) have landed before the CTA can
    // exit; after a timeout the consumers may have stopped waiting for them
    for (uint32_t h = n > static_cast<uint32_t>(NS) ? n - NS : 0u; h < n; ++h)
      mbar_wait_bounded(smem_addr(&full_bar[h % NS]), (h / NS) & 1u, kWaitLimitNs);
    return;
  }

  // ---------------- consumer warps: group grp takes items grp, grp + NG, ...
  // (without a boundary list the ape slice is loaded after the plan scan, so
  // that the scan's loads do not queue behind it)
  if (!ordered) load_ape_regs<TIn>(static_cast<const TIn*>(a.ape), hd, c0, g, cq, ape_r);
  uint32_t local = 0;
  for (uint32_t n = grp; n < items; n += NG, ++local) {
    // one decision for the whole group (also orders the reuse of its reduction buffers)
    if (group_any(grp, NCG, abort_flag != 0)) break;
    const int stage = static_cast<int>(n % NS);
    const uint32_t phase = (n / NS) & 1u;
    // (prefill: the tile's record is requested before the wait for the tile)
    bool ok = true;
    uint32_t e = 0, ragged = 0;
    size_t orow;
    if constexpr (kDecode) {
      orow = own[n].x;
      ok = own[n].x != kInvalidU32;
    } else {
      e = first + n * stride;
      int bl = 0;
      int64_t rp0 = 0;
      bool bad;
      ok = prefill_record(a, e, ragged, bl, rp0, bad);
      orow = token ? ragged : e;
    }
    if (!wait_for<kShortWaits>(smem_addr(&full_bar[stage]), phase, a.wait_ns)) {
      status_or(a.d_status, CKV_STATUS_TIMEOUT);
      abort_flag = 1;
    }
    float* red_l = red_base + (2 * grp + (local & 1u)) * T::RED_FLOATS;
    float* red_a = red_l + 8 * CS;
    if (ok) {
      const TIn* kv_s = reinterpret_cast<const TIn*>(smem + stage * T::TILE_BYTES);
      const TIn* sc_s = kv_s + 128 * CS;
      F2 s[16][2], nml[2];
      float m[4];
      c128_pass1<TIn, CS>(sc_s, g, cq,
                          [&](int k, F2 (&v)[2]) {
                            v[0] = ape_r[k][0];
                            v[1] = ape_r[k][1];
                          },
                          s, m);
      *reinterpret_cast<float4*>(red_l + g * CS + cq) = make_float4(m[0], m[1], m[2], m[3]);
      group_sync(grp, NCG);
      c128_nml<CS>(red_l, cq, nml);
      group_sync(grp, NCG);
      PoolAcc2 acc[2];
      c128_pass2<TIn, CS>(kv_s, g, cq, s, nml, acc);
      store_partials<CS>(red_l, red_a, g, cq, acc);
      group_sync(grp, NCG);
    }
    // the stage is no longer read: hand it back to the producer
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_addr(&empty_bar[stage]));
    if (ok) {
      if (tl < CS) store1<TOut>(out + orow * hd + c0 + tl, finish(tree8(red_a + tl, CS), tree8(red_l + tl, CS)));
      if (token) {  // rows between the previous compress row and this one
        int64_t prev = -1;
        if (e > 0) {
          const ckv_compress_plan_t Q = load_plan_c(a.plan_c + e - 1);
          prev = plan_c_invalid(Q) ? static_cast<int64_t>(ragged) : static_cast<int64_t>(Q.ragged_bl & CKV_RAGGED_MASK);
        }
        zero_rows<CS, TOut, NCG>(out, hd, c0, prev + 1, ragged, tl);
      }
    }
  }
  if (token && first == 0 && grp == 0) {  // rows after the last compress row (and all rows when there is none)
    int64_t last = -1;
    if (num_c > 0) {
      const ckv_compress_plan_t Q = load_plan_c(a.plan_c + num_c - 1);
      last = plan_c_invalid(Q) ? static_cast<int64_t>(a.num_q_tokens) : static_cast<int64_t>(Q.ragged_bl & CKV_RAGGED_MASK);
    }
    zero_rows<CS, TOut, NCG>(out, hd, c0, last + 1, a.num_q_tokens, tl);
  }
}

// ---------------------------------------------------------------- decode (one tile per CTA)
template <typename TIn, typename TOut, bool kShortWaits>
__global__ __launch_bounds__(DecodeCfg<TIn>::THREADS, 6) void c128_decode_kernel(
    const PoolArgs a, uint32_t slices, uint32_t tiles, const __grid_constant__ CUtensorMap page_map) {
  using Cfg = DecodeCfg<TIn>;
  constexpr int CS = Cfg::CS;
  constexpr int NT = Cfg::THREADS;
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t bar_storage;
  TIn* kv_s = reinterpret_cast<TIn*>(smem);
  TIn* sc_s = kv_s + 128 * CS;
  float* red_l = reinterpret_cast<float*>(smem + Cfg::TILE_BYTES);
  float* red_a = red_l + 8 * CS;

  pdl_wait();
  pdl_release();
  const uint32_t tile = blockIdx.x;
  if (tile >= tiles) return;
  const uint32_t b = tile / slices;
  const int c0 = static_cast<int>(tile % slices) * CS;
  const int hd = a.head_dim;
  const size_t width = 2 * static_cast<size_t>(hd);
  const int t = threadIdx.x;
  const TIn* input = static_cast<const TIn*>(a.input);
  TIn* state = static_cast<TIn*>(a.state_mut);
  TOut* out = static_cast<TOut*>(a.out);

  const ckv_decode_plan_t P = load_plan_d(a.plan_d + b);
  if (P.seq_len == kInvalidU32) {
    zero_rows<CS, TOut, NT>(out, hd, c0, b, b + 1, t);
    return;
  }
  const bool boundary = P.seq_len % 128 == 0;
  const int64_t rp0 = P.read_page_0;
  bool ok = P.write_loc >= 0 && static_cast<uint64_t>(P.write_loc) < a.state_rows;
  if (boundary) ok = ok && rp0 >= 0 && static_cast<uint64_t>(rp0) * 128 + 127 < a.state_rows;
  if (!ok) {
    if (t == 0) status_or(a.d_status, CKV_STATUS_BAD_INDEX);
    zero_rows<CS, TOut, NT>(out, hd, c0, b, b + 1, t);
    return;
  }
  const uint32_t bar = smem_addr(&bar_storage);
  if (boundary && t == 0) {
    // slots 0..126 of the page: one 127-row box each for kv and score; the new
    // token (entry 127) comes straight from its input row
    mbar_init(bar, 1);
    fence_mbar_init();
    mbar_arrive_expect_tx(bar, Cfg::TILE_BYTES);
    const int y = static_cast<int>(rp0 * 128);
    tma_box_g2s(smem_addr(kv_s), &page_map, c0, y, bar);
    tma_box_g2s(smem_addr(sc_s), &page_map, hd + c0, y, bar);
    const TIn* row = input + static_cast<size_t>(b) * width;
    bulk_g2s(smem_addr(kv_s + 127 * CS), row + c0, Cfg::SEG_BYTES, bar);
    bulk_g2s(smem_addr(sc_s + 127 * CS), row + hd + c0, Cfg::SEG_BYTES, bar);
  }
  // the new token's slice of kv and score goes to its page slot (never one of
  // the 127 slots read above)
  for (int i = t; i < 2 * Cfg::SEG_BYTES / 16; i += NT) {
    const int half = i / (Cfg::SEG_BYTES / 16);
    const int off = (i % (Cfg::SEG_BYTES / 16)) * (16 / static_cast<int>(sizeof(TIn)));
    const TIn* src = input + static_cast<size_t>(b) * width + half * hd + c0 + off;
    TIn* dst = state + static_cast<size_t>(P.write_loc) * width + half * hd + c0 + off;
    st16(dst, ld_stream16(src));
  }
  if (!boundary) {
    zero_rows<CS, TOut, NT>(out, hd, c0, b, b + 1, t);
    return;
  }
  __syncthreads();  // barrier initialisation is visible to every waiting thread
  const int q = t % Cfg::QUADS;
  const int g = t / Cfg::QUADS;
  const int cq = 4 * q;
  const TIn* ape = static_cast<const TIn*>(a.ape) + static_cast<size_t>(16 * g) * hd + c0 + cq;
  auto ape_at = [&](int k, F2 (&v)[2]) { ldg4x2<TIn>(ape + static_cast<size_t>(k) * hd, v); };
  if (!wait_for<kShortWaits>(bar, 0, a.wait_ns)) {
    status_or(a.d_status, CKV_STATUS_TIMEOUT);
    mbar_wait_bounded(bar, 0, kWaitLimitNs);  // let copies in flight land before the CTA can exit
  }
  float m[4];
  F2 nml[2];
  c128_max_only<TIn, CS>(sc_s, g, cq, ape_at, m);
  *reinterpret_cast<float4*>(red_l + g * CS + cq) = make_float4(m[0], m[1], m[2], m[3]);
  __syncthreads();
  c128_nml<CS>(red_l, cq, nml);
  __syncthreads();
  PoolAcc2 acc[2];
  c128_pass2_recompute<TIn, CS>(kv_s, sc_s, g, cq, ape_at, nml, acc);
  store_partials<CS>(red_l, red_a, g, cq, acc);
  __syncthreads();
  if (t < CS) store1<TOut>(out + static_cast<size_t>(b) * hd + c0 + t, finish(tree8(red_a + t, CS), tree8(red_l + t, CS)));
}

// ---------------------------------------------------------------- tensor maps
// A [rows, cols] row-major tensor read in boxes of [box_rows, box_cols].
int make_map(CUtensorMap* map, const void* base, int dtype, uint64_t cols, uint64_t rows, uint32_t box_cols,
             uint32_t box_rows) {
  const uint64_t esz = dtype == CKV_BF16 ? 2 : 4;
  const uint64_t dims[2] = {cols, rows};
  const uint64_t strides[1] = {cols * esz};
  const uint32_t box[2] = {box_cols, box_rows};
  return encode_tensor_map(map, dtype, 2, base, dims, strides, box);
}

// ---------------------------------------------------------------- launchers
// `configured` is a per-device cache (atomics: a repeated set-up by racing
// threads is harmless).
template <typename K>
int opt_in_smem(K kernel, int bytes, std::atomic<bool>* configured) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return CKV_ERR_LAUNCH;
  const bool cached_dev = dev >= 0 && dev < 64;
  if (!cached_dev || !configured[dev].load(std::memory_order_acquire)) {
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess) {
      cudaGetLastError();
      return CKV_ERR_LAUNCH;
    }
    if (cached_dev) configured[dev].store(true, std::memory_order_release);
  }
  return CKV_OK;
}

template <typename TIn, typename TOut, bool kShortWaits>
int launch_prefill_t(const PoolArgs& a, cudaStream_t s) {
  constexpr int CS = sizeof(TIn) == 2 ? 128 : 64;
  constexpr int NS = 3;
  using Cfg = PersistCfg<TIn, CS, NS, 1, false>;
  const uint32_t slices = static_cast<uint32_t>(a.head_dim / CS);
  const bool token = a.out_layout == CKV_OUT_TOKEN;
  if (a.capacity == 0 && !(token && a.num_q_tokens > 0)) return CKV_OK;
  static std::atomic<bool> configured[64];
  auto kernel = c128_persistent_kernel<TIn, TOut, CS, NS, 1, false, kShortWaits>;
  int rc = opt_in_smem(kernel, Cfg::SMEM, configured);
  if (rc) return rc;
  // one persistent CTA per SM; every CTA serves one channel slice
  const uint32_t per_slice = std::max<uint32_t>(
      1, std::min<uint32_t>(static_cast<uint32_t>(sm_count()) / slices, std::max<uint32_t>(a.capacity, 1)));
  // tensor-map row coordinates are 32-bit
  if (a.state_rows > 0x7FFFFFFFull) return CKV_ERR_SIZE;
  alignas(64) CUtensorMap in_map;
  alignas(64) GatherMaps gather;
  memset(&in_map, 0, sizeof in_map);
  memset(&gather, 0, sizeof gather);
  if (a.num_q_tokens > 0) {
    rc = make_map(&in_map, a.input, a.in_dtype, 2ull * a.head_dim, a.num_q_tokens, CS, 128);
    for (int k = 0; k < 4 && !rc; ++k)
      rc = make_map(&gather.input[k], a.input, a.in_dtype, 2ull * a.head_dim, a.num_q_tokens, CS,
                    gather_height(k));
    if (rc) return rc;
  }
  if (a.state_rows > 0) {
    for (int k = 0; k < 4 && !rc; ++k)
      rc = make_map(&gather.state[k], a.state, a.in_dtype, 2ull * a.head_dim, a.state_rows, CS, gather_height(k));
    if (rc) return rc;
  }
  return launch_pdl(kernel, dim3(per_slice * slices), dim3(Cfg::THREADS), Cfg::SMEM, s, a, slices, in_map, in_map,
                    gather);
}

// Persistent decode tiles: kDecCS channels (bf16; half for fp32) x 127 page
// rows, kDecNS stages, kDecNG consumer groups.
constexpr int kDecCS = 64;
constexpr int kDecNS = 4;
static_assert(kDecLag < kDecNS, "the paced wait must name a stage that is not being refilled");
constexpr int kDecNG = 2;  // consumer groups reduce alternate tiles

template <typename TIn, typename TOut, bool kShortWaits>
int launch_decode_t(const PoolArgs& a, cudaStream_t s) {
  if (a.capacity == 0) return CKV_OK;
  if (a.state_rows == 0 || a.state_rows > 0x7FFFFFFFull) return CKV_ERR_SIZE;
  constexpr int PCS = sizeof(TIn) == 2 ? kDecCS : kDecCS / 2;
  const uint32_t pslices = static_cast<uint32_t>(a.head_dim / PCS);
  const uint32_t per_slice = std::max<uint32_t>(1, static_cast<uint32_t>(sm_count()) / pslices);
  // each CTA owns at most ceil(batch / per_slice) boundary rows and
  // ceil(batch / grid) rows without a window: both lists live in shared memory
  if ((a.capacity + per_slice - 1) / per_slice <= static_cast<uint32_t>(kOwnRows)) {
    // persistent: every CTA scans the plan and streams its share of boundary tiles
    alignas(64) CUtensorMap page_map;
    int rc = make_map(&page_map, a.state_mut, a.in_dtype, 2ull * a.head_dim, a.state_rows, PCS, 127);
    if (rc) return rc;
    using Cfg = PersistCfg<TIn, PCS, kDecNS, kDecNG, true>;
    static std::atomic<bool> configured_p[64];
    auto kernel = c128_persistent_kernel<TIn, TOut, PCS, kDecNS, kDecNG, true, kShortWaits>;
    rc = opt_in_smem(kernel, Cfg::SMEM, configured_p);
    if (rc) return rc;
    return launch_pdl(kernel, dim3(per_slice * pslices), dim3(Cfg::THREADS), Cfg::SMEM, s, a, pslices, page_map,
                      page_map, GatherMaps{});
  }
  // very large batches: one CTA per (row, slice)
  constexpr int CS = DecodeCfg<TIn>::CS;
  const uint32_t slices = static_cast<uint32_t>(a.head_dim / CS);
  alignas(64) CUtensorMap page_map;
  int rc = make_map(&page_map, a.state_mut, a.in_dtype, 2ull * a.head_dim, a.state_rows, CS, 127);
  if (rc) return rc;
  using Cfg = DecodeCfg<TIn>;
  const uint64_t tiles64 = static_cast<uint64_t>(a.capacity) * slices;
  if (tiles64 > 0x7FFFFFFFull) return CKV_ERR_SIZE;
  static std::atomic<bool> configured[64];
  auto kernel = c128_decode_kernel<TIn, TOut, kShortWaits>;
  rc = opt_in_smem(kernel, Cfg::SMEM, configured);
  if (rc) return rc;
  const uint32_t tiles = static_cast<uint32_t>(tiles64);
  return launch_pdl(kernel, dim3(tiles), dim3(Cfg::THREADS), Cfg::SMEM, s, a, slices, tiles, page_map);
}

template <bool kDecode, typename TIn, typename TOut>
int launch_t(const PoolArgs& a, cudaStream_t s) {
  // kernels built for waits shorter than try_wait's window only for such limits
  if (a.wait_ns < kShortWaitNs)
    return kDecode ? launch_decode_t<TIn, TOut, true>(a, s) : launch_prefill_t<TIn, TOut, true>(a, s);
  return kDecode ? launch_decode_t<TIn, TOut, false>(a, s) : launch_prefill_t<TIn, TOut, false>(a, s);
}

template <bool kDecode>
int dispatch(const PoolArgs& a, cudaStream_t s) {
  if (a.in_dtype == CKV_BF16) {
    if (a.out_dtype == CKV_BF16) return launch_t<kDecode, __nv_bfloat16, __nv_bfloat16>(a, s);
    return launch_t<kDecode, __nv_bfloat16, float>(a, s);
  }
  if (a.out_dtype == CKV_BF16) return launch_t<kDecode, float, __nv_bfloat16>(a, s);
  return launch_t<kDecode, float, float>(a, s);
}

}  // namespace

int launch_c128_pool_prefill(const PoolArgs& a, cudaStream_t s) { return dispatch<false>(a, s); }

namespace {
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// Fetched once, by the first caller (a function-local static: its
// initialisation is thread-safe).
EncodeTiledFn encoder() {
  static const EncodeTiledFn fn = []() -> EncodeTiledFn {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<EncodeTiledFn>(p);
    cudaGetLastError();
    return nullptr;
  }();
  return fn;
}
}  // namespace

int encode_tensor_map(CUtensorMap* map, int dtype, uint32_t rank, const void* base, const uint64_t* dims,
                      const uint64_t* strides_bytes, const uint32_t* box) {
  EncodeTiledFn fn = encoder();
  if (fn == nullptr || rank < 1 || rank > 5) return CKV_ERR_LAUNCH;
  cuuint64_t d[5], st[4];
  cuuint32_t b[5], estr[5];
  for (uint32_t i = 0; i < rank; ++i) {
    d[i] = dims[i];
    b[i] = box[i];
    estr[i] = 1;
    if (i + 1 < rank) st[i] = strides_bytes[i];
  }
  const CUresult r = fn(map, dtype == CKV_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                        rank, const_cast<void*>(base), d, st, b, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? CKV_OK : CKV_ERR_LAUNCH;
}
int launch_c128_decode(const PoolArgs& a, cudaStream_t s) { return dispatch<true>(a, s); }

}  // namespace ckv
