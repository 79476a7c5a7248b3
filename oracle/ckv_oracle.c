/*
 * ckv_oracle.c -- CPU oracle for the compressed-KV compressor (C4 / C128).
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, plain, obviously-correct
 * statement of what the GPU library computes.  It is used by the test-suite,
 * by the smoke check and by the benchmark's CPU-baseline leg, and by nothing
 * else.  It shares no code, header, table or constant generator with the CUDA
 * library: every layout it needs (the plan records, the dtype codes) is
 * restated here from the pages it cites.
 *
 * Sources (SGLang, DeepSeek-V4 compressor):
 *   [c_plan]  python/sglang/jit_kernel/csrc/deepseek_v4/c_plan.cuh
 *   [cv2]     python/sglang/srt/layers/attention/dsv4/compressor_v2.py
 *   [c4]      python/sglang/jit_kernel/csrc/deepseek_v4/c4.cuh
 *
 * Arithmetic: single-threaded loops; the per-channel score s_i = score + ape is
 * rounded in fp32 (as both [c4] c4_forward and the [cv2] C128 kernels do),
 * everything after it (max, exp, sums, division) is carried in double and the
 * result is rounded once to the output dtype (RNE).
 *
 * Compile with -O2 -ffp-contract=off (no fast-math) so that no fused
 * multiply-add or reassociation changes the double arithmetic.
 */
#include <math.h>
#include <stdint.h>

#include <stdlib.h>
#include <string.h>

/* ----- dtype codes and layouts (a format both sides must agree on) ------- */
enum { ORC_F32 = 0, ORC_BF16 = 1 };
enum { ORC_OUT_TOKEN = 0, ORC_OUT_COMPACT = 1 };

/* Error returns of the oracle (host-side validation, [c_plan] RuntimeCheck). */
enum {
  ORC_OK = 0,
  ORC_BAD_RATIO = -1,
  ORC_BAD_HEAD_DIM = -2,
  ORC_BAD_BATCH = -3,
  ORC_BAD_DTYPE = -5,
  ORC_BAD_LENGTH = -8,
  ORC_BAD_TOTAL = -9,
  ORC_CAPACITY = -10,
  ORC_BAD_INDEX = -11,
};

/* CompressPlan, 16 bytes ([c_plan] plan_compress_prefill, CPU loop; fields
 * seq_len / ragged_id / buffer_len / read_page_0 / read_page_1).  The ragged id
 * is widened to 24 bits and shares its word with the 8-bit buffer_len
 * (buffer_len <= 127 because the window is at most 128). */
typedef struct {
  uint32_t seq_len;
  uint32_t ragged_bl; /* ragged_id | buffer_len << 24 */
  int32_t read_page_0;
  int32_t read_page_1;
} orc_plan_c;

/* WritePlan, 8 bytes: {ragged_id, write_loc} ([c_plan] pack_w / legacy kernel). */
typedef struct {
  uint32_t ragged_id;
  int32_t write_loc;
} orc_plan_w;

/* DecodePlan, 16 bytes ([c_plan] plan_compress_decode_legacy_kernel). */
typedef struct {
  uint32_t seq_len;
  int32_t write_loc;
  int32_t read_page_0;
  int32_t read_page_1;
} orc_plan_d;

/* ----- scalar helpers ---------------------------------------------------- */
static float bf16_bits_to_float(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

/* Round a double to bfloat16 (8 significant bits, fp32 exponent range) once,
 * to nearest, ties to even.  Written from the format's definition: find the
 * spacing q of bf16 numbers at |x| (2^(e-7) for |x| in [2^e, 2^(e+1)), never
 * below the subnormal spacing 2^-133) and round x/q to an integer with
 * nearbyint (default rounding mode = nearest-even). */
static uint16_t double_to_bf16_bits(double x) {
  if (isnan(x)) return 0x7FC0;
  uint16_t sign = signbit(x) ? 0x8000u : 0u;
  double a = fabs(x);
  if (a == 0.0) return sign;
  if (isinf(a)) return (uint16_t)(sign | 0x7F80u);
  int k;
  frexp(a, &k); /* a = f * 2^k, f in [0.5, 1): a in [2^(k-1), 2^k) */
  int qexp = (k - 1) - 7;
  if (qexp < -133) qexp = -133;
  double r = ldexp(nearbyint(ldexp(a, -qexp)), qexp);
  if (r >= 0x1p128) return (uint16_t)(sign | 0x7F80u);
  float f = (float)r; /* exact: r has at most 8 significant bits */
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  return (uint16_t)(sign | ((u >> 16) & 0x7FFFu));
}

static float load_elem(const void* base, size_t idx, int dtype) {
  if (dtype == ORC_BF16) return bf16_bits_to_float(((const uint16_t*)base)[idx]);
  return ((const float*)base)[idx];
}

static void store_elem(void* base, size_t idx, int dtype, double v) {
  if (dtype == ORC_BF16)
    ((uint16_t*)base)[idx] = double_to_bf16_bits(v);
  else
    ((float*)base)[idx] = (float)v;
}

static size_t elem_size(int dtype) { return dtype == ORC_BF16 ? 2 : 4; }

static int window_of(int ratio) { return ratio == 4 ? 8 : ratio; }

/* Width of one kv_score row: C4 = | kv-overlap | kv | score-overlap | score |
 * (4*hd, [c4] Compress4DecodeParams); C128 = | kv | score | (2*hd, [cv2]
 * _compress_forward_c128_fallback). */
static int row_width(int ratio, int hd) { return ratio == 4 ? 4 * hd : 2 * hd; }

/* Legacy per-request state addressing ([c_plan] plan_compress_*_legacy_kernel):
 *   C4:   page = rid*2 + (position/4) % 2, slot = page*4 + position % 4
 *   C128: page = rid,                      slot = rid*128 + position % 128 */
static int64_t legacy_page(int ratio, int64_t rid, int64_t position) {
  if (ratio == 4) return rid * 2 + ((position / 4) & 1);
  return rid;
}

static int64_t legacy_loc(int ratio, int64_t rid, int64_t position) {
  return legacy_page(ratio, rid, position) * ratio + position % ratio;
}

/* ----- the pooling step -------------------------------------------------- */
/* One compressed row from a window of W entries ([c4] c4_forward, [cv2]
 * _compress_forward_c128_fallback):
 *   for every channel c:
 *     s_i = fp32(score_i[c]) + fp32(ape[i][c])          (rounded in fp32)
 *     out[c] = sum_i kv_i[c] * exp(s_i - m) / sum_i exp(s_i - m),  m = max_i s_i
 * entries[i] points at the start of the kv_score row that holds window entry i,
 * or is NULL for an entry that is masked out (C4, first group: [c4] c4_forward
 * sets kv = 0 and score = -1e9 there, whose weight exp(-1e9 - m) is exactly 0).
 * C4 columns: entries 0..3 are the previous group, read from the overlap halves
 * (kv at [0,hd), score at [2hd,3hd)); entries 4..7 read the main halves (kv at
 * [hd,2hd), score at [3hd,4hd)).  C128 columns: kv at [0,hd), score at [hd,2hd).
 * The ape row is the window index i. */
static void pool_window(int ratio, int hd, int in_dtype, int out_dtype, const void* const* entries,
                        const void* ape, void* out_row) {
  const int W = window_of(ratio);
  float* s = (float*)malloc(sizeof(float) * (size_t)W);
  for (int c = 0; c < hd; ++c) {
    int have = 0;
    float m = 0.0f;
    for (int i = 0; i < W; ++i) {
      if (!entries[i]) continue;
      int sc_col = ratio == 4 ? (i < 4 ? 2 * hd : 3 * hd) + c : hd + c;
      float score = load_elem(entries[i], (size_t)sc_col, in_dtype);
      int arow = i;
      float bias = load_elem(ape, (size_t)arow * hd + c, in_dtype);
      float si = score + bias; /* one fp32 rounding */
      s[i] = si;
      if (!have || si > m) m = si;
      have = 1;
    }
    double num = 0.0, den = 0.0;
    for (int i = 0; i < W; ++i) {
      if (!entries[i]) continue;
      int kv_col = (ratio == 4) ? (i < 4 ? 0 : hd) + c : c;
      double kv = (double)load_elem(entries[i], (size_t)kv_col, in_dtype);
      double w = exp((double)s[i] - (double)m);
      num += kv * w;
      den += w;
    }
    store_elem(out_row, (size_t)c, out_dtype, have ? num / den : 0.0);
  }
  free(s);
}

static const void* row_ptr(const void* base, int64_t row, int width, int dtype) {
  return (const char*)base + (size_t)row * (size_t)width * elem_size(dtype);
}

static int check_common(int ratio, int hd, int in_dtype, int out_dtype) {
  if (ratio != 4 && ratio != 128) return ORC_BAD_RATIO;
  if (hd <= 0 || hd % 128 != 0 || hd > 1024) return ORC_BAD_HEAD_DIM;
  if ((in_dtype != ORC_F32 && in_dtype != ORC_BF16) || (out_dtype != ORC_F32 && out_dtype != ORC_BF16))
    return ORC_BAD_DTYPE;
  return ORC_OK;
}

/* ----- plans -------------------------------------------------------------- */

/* Decode plan, one row per request ([c_plan] plan_compress_decode_legacy_kernel):
 *   position_1 = seq_len - 1, position_0 = max(position_1 - ratio, 0)
 *   write_loc = slot(rid, position_1), read_page_0/1 = page(rid, position_0/1). */
int orc_plan_decode(int ratio, const int64_t* rid, const int64_t* seq_lens, uint32_t batch, void* plan_d_out) {
  if (ratio != 4 && ratio != 128) return ORC_BAD_RATIO;
  orc_plan_d* plan = (orc_plan_d*)plan_d_out;
  for (uint32_t b = 0; b < batch; ++b) {
    if (seq_lens[b] < 1 || seq_lens[b] > INT32_MAX || rid[b] < 0) return ORC_BAD_LENGTH;
    int64_t p1 = seq_lens[b] - 1;
    int64_t p0 = p1 - ratio > 0 ? p1 - ratio : 0;
    int64_t loc = legacy_loc(ratio, rid[b], p1);
    if (loc > INT32_MAX) return ORC_BAD_INDEX;
    plan[b].seq_len = (uint32_t)seq_lens[b];
    plan[b].write_loc = (int32_t)loc;
    plan[b].read_page_0 = (int32_t)legacy_page(ratio, rid[b], p0);
    plan[b].read_page_1 = (int32_t)legacy_page(ratio, rid[b], p1);
  }
  return ORC_OK;
}

/* Prefill plans: the sequential CPU loop of [c_plan] plan_compress_prefill_legacy
 * (one request after another, positions ascending), followed by the legacy slot
 * translation of plan_compress_prefill_legacy_kernel.  For request b with
 * prefix pl = seq_len - extend_len and extend token j (position p = pl + j,
 * ragged id = tokens before b + j):
 *   compress iff (p + 1) % ratio == 0:
 *       {seq_len = p+1, ragged_id, buffer_len = W - min(j+1, W),
 *        read_page_0 = page(rid, max(p - ratio, 0)), read_page_1 = page(rid, p)}
 *   write    iff p >= (seq_len/ratio)*ratio - (ratio == 4 ? 4 : 0):
 *       {ragged_id, write_loc = slot(rid, p)}
 * Entries [count, capacity) are filled with the invalid record (all bytes 0xFF)
 * when pad_invalid is set.  counts[0] = compress entries, counts[1] = writes. */
int orc_plan_prefill(int ratio, const int64_t* rid, const int64_t* seq_lens, const int64_t* extend_lens,
                     uint32_t batch, uint32_t num_q_tokens, uint32_t cap_c, uint32_t cap_w, int pad_invalid,
                     void* plan_c_out, void* plan_w_out, uint32_t* counts) {
  if (ratio != 4 && ratio != 128) return ORC_BAD_RATIO;
  if (batch > 1024) return ORC_BAD_BATCH;
  if (num_q_tokens >= (1u << 24)) return ORC_BAD_BATCH;
  const int W = window_of(ratio);
  const int64_t overlap = ratio == 4 ? 4 : 0;
  orc_plan_c* pc = (orc_plan_c*)plan_c_out;
  orc_plan_w* pw = (orc_plan_w*)plan_w_out;
  uint64_t token_base = 0, nc = 0, nw = 0;
  for (uint32_t b = 0; b < batch; ++b) {
    const int64_t sl = seq_lens[b], el = extend_lens[b];
    if (!(0 < el && el <= sl) || sl > INT32_MAX || rid[b] < 0) return ORC_BAD_LENGTH;
    const int64_t pl = sl - el;
    const int64_t first_w = (sl / ratio) * ratio - overlap;
    for (int64_t j = 0; j < el; ++j) {
      const int64_t p = pl + j;
      const uint64_t ragged = token_base + (uint64_t)j;
      if ((p + 1) % ratio == 0) {
        if (nc < cap_c) {
          const int64_t bl = W - (j + 1 < W ? j + 1 : W);
          const int64_t p0 = p - ratio > 0 ? p - ratio : 0;
          pc[nc].seq_len = (uint32_t)(p + 1);
          pc[nc].ragged_bl = (uint32_t)ragged | ((uint32_t)bl << 24);
          pc[nc].read_page_0 = (int32_t)legacy_page(ratio, rid[b], p0);
          pc[nc].read_page_1 = (int32_t)legacy_page(ratio, rid[b], p);
        }
        ++nc;
      }
      if (p >= first_w) {
        if (nw < cap_w) {
          pw[nw].ragged_id = (uint32_t)ragged;
          pw[nw].write_loc = (int32_t)legacy_loc(ratio, rid[b], p);
        }
        ++nw;
      }
    }
    token_base += (uint64_t)el;
  }
  counts[0] = (uint32_t)nc;
  counts[1] = (uint32_t)nw;
  if (token_base != num_q_tokens) return ORC_BAD_TOTAL;
  if (nc > cap_c || nw > cap_w) return ORC_CAPACITY;
  if (pad_invalid) {
    if (cap_c > nc) memset(pc + nc, 0xFF, sizeof(orc_plan_c) * (cap_c - nc));
    if (cap_w > nw) memset(pw + nw, 0xFF, sizeof(orc_plan_w) * (cap_w - nw));
  }
  return ORC_OK;
}

/* ----- SWA-paged plans ([c_plan] plan_compress_prefill / _decode, main path) */

/* State row of position p of request rid through the SWA mapping ([c_plan]
 * compute_loc): swa = full_to_state[req_to_token[rid][p]], row =
 * (swa / swa_page_size) * ring_size + swa % ring_size.  -1 when a map entry is
 * out of range. */
static int64_t paged_row(const int32_t* r2t, int64_t stride, const int64_t* f2s, uint64_t nfull, int32_t sps,
                         int32_t ring, int64_t rid, int64_t p) {
  const int32_t raw = r2t[rid * stride + p];
  if (raw < 0 || (uint64_t)raw >= nfull) return -1;
  const int64_t swa = f2s[raw];
  if (swa < 0) return -1;
  return (swa / sps) * ring + swa % ring;
}

/* State row of position p under the paged addressing: C4 through the SWA
 * mapping (paged_row), C128 request-scoped rid * ring + p % ring ([c_plan]
 * compute_c128_loc). */
static int64_t paged_or_c128_row(int ratio, const int32_t* r2t, int64_t stride, const int64_t* f2s, uint64_t nfull,
                                 int32_t sps, int32_t ring, int64_t rid, int64_t p) {
  if (ratio == 128) return rid * ring + p % ring;
  return paged_row(r2t, stride, f2s, nfull, sps, ring, rid, p);
}

/* Prefill plans with SWA-paged state: the CPU loop of [c_plan]
 * plan_compress_prefill (C4 writes every p >= first_w and, as the ratio
 * overlaps, the last ratio positions of every SWA page), with first_w =
 * min((sl/R)*R - (C4 ? 4 : 0), sl - mtp_pad), mtp_pad = min(ring - R, 4) as the
 * GPU-input planner has it; then kernel_1's translation of positions into
 * rows and pages, which it applies to compress records with buffer_len > 0
 * only -- the others keep read_page_0 = -1, read_page_1 = batch index.
 * C128 needs ring 128 (its pooling reads the window from read_page_0). */
int orc_plan_prefill_paged(int ratio, const int64_t* rid, const int32_t* r2t, int64_t stride, uint32_t num_reqs,
                           const int64_t* f2s, uint64_t nfull, int32_t sps, int32_t ring, const int64_t* seq_lens,
                           const int64_t* extend_lens, uint32_t batch, uint32_t num_q_tokens, uint32_t cap_c,
                           uint32_t cap_w, int pad_invalid, void* plan_c_out, void* plan_w_out, uint32_t* counts) {
  if (ratio != 4 && ratio != 128) return ORC_BAD_RATIO;
  if (batch > 1024 || num_q_tokens >= (1u << 24)) return ORC_BAD_BATCH;
  if (ratio == 128 && ring != 128) return ORC_BAD_BATCH;
  if (ratio == 4 && (sps <= 0 || ring < 8 || ring % 4 || sps % ring)) return ORC_BAD_BATCH;
  const int W = ratio == 4 ? 8 : 128;
  const int64_t mtp_pad = ring - ratio < 4 ? ring - ratio : 4;
  orc_plan_c* pc = (orc_plan_c*)plan_c_out;
  orc_plan_w* pw = (orc_plan_w*)plan_w_out;
  uint64_t token_base = 0, nc = 0, nw = 0;
  for (uint32_t b = 0; b < batch; ++b) {
    const int64_t sl = seq_lens[b], el = extend_lens[b];
    if (!(0 < el && el <= sl) || sl > INT32_MAX || rid[b] < 0) return ORC_BAD_LENGTH;
    if (ratio == 4 && ((uint64_t)rid[b] >= num_reqs || sl > stride)) return ORC_BAD_INDEX;
    const int64_t pl = sl - el;
    int64_t first_w = (sl / ratio) * ratio - (ratio == 4 ? 4 : 0);
    if (sl - mtp_pad < first_w) first_w = sl - mtp_pad;
    for (int64_t j = 0; j < el; ++j) {
      const int64_t p = pl + j;
      const uint64_t ragged = token_base + (uint64_t)j;
      if ((p + 1) % ratio == 0) {
        if (nc < cap_c) {
          const int64_t bl = W - (j + 1 < W ? j + 1 : W);
          int64_t page0 = -1, page1 = b;
          if (bl > 0) {
            const int64_t p0 = p - ratio > 0 ? p - ratio : 0;
            const int64_t row0 = paged_or_c128_row(ratio, r2t, stride, f2s, nfull, sps, ring, rid[b], p0);
            const int64_t row1 = paged_or_c128_row(ratio, r2t, stride, f2s, nfull, sps, ring, rid[b], p);
            if (row0 < 0 || row1 < 0) return ORC_BAD_INDEX;
            page0 = row0 / ratio;
            page1 = row1 / ratio;
          }
          pc[nc].seq_len = (uint32_t)(p + 1);
          pc[nc].ragged_bl = (uint32_t)ragged | ((uint32_t)bl << 24);
          pc[nc].read_page_0 = (int32_t)page0;
          pc[nc].read_page_1 = (int32_t)page1;
        }
        ++nc;
      }
      if (p >= first_w || (ratio == 4 && p % sps >= sps - ratio)) {
        if (nw < cap_w) {
          const int64_t row = paged_or_c128_row(ratio, r2t, stride, f2s, nfull, sps, ring, rid[b], p);
          if (row < 0) return ORC_BAD_INDEX;
          pw[nw].ragged_id = (uint32_t)ragged;
          pw[nw].write_loc = (int32_t)row;
        }
        ++nw;
      }
    }
    token_base += (uint64_t)el;
  }
  counts[0] = (uint32_t)nc;
  counts[1] = (uint32_t)nw;
  if (token_base != num_q_tokens) return ORC_BAD_TOTAL;
  if (nc > cap_c || nw > cap_w) return ORC_CAPACITY;
  if (pad_invalid) {
    if (cap_c > nc) memset(pc + nc, 0xFF, sizeof(orc_plan_c) * (cap_c - nc));
    if (cap_w > nw) memset(pw + nw, 0xFF, sizeof(orc_plan_w) * (cap_w - nw));
  }
  return ORC_OK;
}

/* Decode plan with SWA-paged state ([c_plan] plan_compress_decode_kernel):
 * write_loc = row of position seq_len-1, read pages = rows of positions
 * max(seq_len-1-4, 0) and seq_len-1, divided by 4.  C128 with its 128-row ring
 * (compute_c128_loc) is the legacy plan. */
int orc_plan_decode_paged(int ratio, const int64_t* rid, const int32_t* r2t, int64_t stride, uint32_t num_reqs,
                          const int64_t* f2s, uint64_t nfull, int32_t sps, int32_t ring, const int64_t* seq_lens,
                          uint32_t batch, void* plan_d_out) {
  if (ratio == 128) return ring == 128 ? orc_plan_decode(ratio, rid, seq_lens, batch, plan_d_out) : ORC_BAD_BATCH;
  if (ratio != 4) return ORC_BAD_RATIO;
  if (sps <= 0 || ring < 8 || ring % 4 || sps % ring) return ORC_BAD_BATCH;
  orc_plan_d* plan = (orc_plan_d*)plan_d_out;
  for (uint32_t b = 0; b < batch; ++b) {
    if (seq_lens[b] < 1 || seq_lens[b] > INT32_MAX || rid[b] < 0) return ORC_BAD_LENGTH;
    if ((uint64_t)rid[b] >= num_reqs || seq_lens[b] > stride) return ORC_BAD_INDEX;
    const int64_t p1 = seq_lens[b] - 1;
    const int64_t p0 = p1 - 4 > 0 ? p1 - 4 : 0;
    const int64_t row1 = paged_row(r2t, stride, f2s, nfull, sps, ring, rid[b], p1);
    const int64_t row0 = paged_row(r2t, stride, f2s, nfull, sps, ring, rid[b], p0);
    if (row0 < 0 || row1 < 0) return ORC_BAD_INDEX;
    plan[b].seq_len = (uint32_t)seq_lens[b];
    plan[b].write_loc = (int32_t)row1;
    plan[b].read_page_0 = (int32_t)(row0 / 4);
    plan[b].read_page_1 = (int32_t)(row1 / 4);
  }
  return ORC_OK;
}

/* ----- the compute steps ------------------------------------------------- */

/* Prefill pooling, one compressed row per compress-plan entry ([c4]
 * flash_c4_prefill<kWrite=false> + c4_forward; [cv2] C128 fallback, with the
 * window read the way c4_forward reads it): window entry i of the event ending
 * at position p = seq_len-1 is position p - W + 1 + i; it comes from the state
 * when i < buffer_len and from ragged input row ragged_id - (W-1) + i otherwise.
 * State rows: C4 entry i lives in page (i < 4 ? read_page_0 : read_page_1),
 * slot i % 4; C128 entry i lives in page read_page_0, slot i.
 * Output: token layout writes row ragged_id of a zero-filled [num_q_tokens, hd]
 * tensor; compact layout writes row e of [num_c, hd] in plan order.
 * This step only reads the state (the writes come after it, [c4] run_prefill). */
int orc_compress_pool_prefill(int ratio, int hd, int in_dtype, int out_dtype, const void* state,
                              uint64_t state_rows, const void* input, uint32_t num_q_tokens, const void* ape,
                              const void* plan_c_in, uint32_t num_c, int out_layout, void* out) {
  int rc = check_common(ratio, hd, in_dtype, out_dtype);
  if (rc) return rc;
  const int W = window_of(ratio);
  const int width = row_width(ratio, hd);
  const orc_plan_c* pc = (const orc_plan_c*)plan_c_in;
  const size_t out_rows = out_layout == ORC_OUT_TOKEN ? num_q_tokens : num_c;
  memset(out, 0, out_rows * (size_t)hd * elem_size(out_dtype));
  const void** entries = (const void**)malloc(sizeof(void*) * (size_t)W);
  for (uint32_t e = 0; e < num_c; ++e) {
    const orc_plan_c* P = &pc[e];
    if (P->seq_len == 0xFFFFFFFFu) continue; /* invalid (padding) entry */
    const int64_t ragged = P->ragged_bl & 0x00FFFFFFu;
    const int bl = (int)(P->ragged_bl >> 24);
    const int64_t seq_len = P->seq_len;
    if (ragged >= num_q_tokens) { free(entries); return ORC_BAD_INDEX; }
    for (int i = 0; i < W; ++i) {
      if (ratio == 4 && seq_len == 4 && i < 4) { /* first group: no previous group */
        entries[i] = NULL;
        continue;
      }
      if (i < bl) {
        int64_t srow = ratio == 4 ? (int64_t)(i < 4 ? P->read_page_0 : P->read_page_1) * 4 + i % 4
                                  : (int64_t)P->read_page_0 * 128 + i;
        if (srow < 0 || (uint64_t)srow >= state_rows) { free(entries); return ORC_BAD_INDEX; }
        entries[i] = row_ptr(state, srow, width, in_dtype);
      } else {
        int64_t irow = ragged - (W - 1) + i;
        if (irow < 0) { free(entries); return ORC_BAD_INDEX; }
        entries[i] = row_ptr(input, irow, width, in_dtype);
      }
    }
    size_t orow = out_layout == ORC_OUT_TOKEN ? (size_t)ragged : (size_t)e;
    void* dst = (char*)out + orow * (size_t)hd * elem_size(out_dtype);
    pool_window(ratio, hd, in_dtype, out_dtype, (const void* const*)entries, ape, dst);
  }
  free(entries);
  return ORC_OK;
}

/* Prefill state write ([c4] c4_write, [cv2] _c128_compress_prefill_write_kernel):
 * state[write_loc] = input[ragged_id], the whole row, bit for bit. */
int orc_compress_write(int ratio, int hd, int dtype, void* state, uint64_t state_rows, const void* input,
                       uint32_t num_q_tokens, const void* plan_w_in, uint32_t num_w) {
  if (ratio != 4 && ratio != 128) return ORC_BAD_RATIO;
  const int width = row_width(ratio, hd);
  const size_t row_bytes = (size_t)width * elem_size(dtype);
  const orc_plan_w* pw = (const orc_plan_w*)plan_w_in;
  for (uint32_t k = 0; k < num_w; ++k) {
    if (pw[k].write_loc < 0 || pw[k].ragged_id == 0xFFFFFFFFu) continue;
    if (pw[k].ragged_id >= num_q_tokens || (uint64_t)pw[k].write_loc >= state_rows) return ORC_BAD_INDEX;
    memcpy((char*)state + (size_t)pw[k].write_loc * row_bytes, row_ptr(input, pw[k].ragged_id, width, dtype),
           row_bytes);
  }
  return ORC_OK;
}

/* Decode ([c4] flash_c4_decode, [cv2] _c128_compress_decode_kernel and the
 * fallback): write the new row to state[write_loc]; when seq_len % ratio == 0
 * pool the W-entry window, all of it now in the state (C4 entry i: page
 * read_page_0 for i < 4 else read_page_1, slot i % 4; C128: page read_page_0,
 * slot i); otherwise the output row is zero. */
int orc_compress_decode(int ratio, int hd, int in_dtype, int out_dtype, void* state, uint64_t state_rows,
                        const void* input, const void* ape, const void* plan_d_in, uint32_t batch, void* out) {
  int rc = check_common(ratio, hd, in_dtype, out_dtype);
  if (rc) return rc;
  const int W = window_of(ratio);
  const int width = row_width(ratio, hd);
  const size_t row_bytes = (size_t)width * elem_size(in_dtype);
  const orc_plan_d* pd = (const orc_plan_d*)plan_d_in;
  memset(out, 0, (size_t)batch * (size_t)hd * elem_size(out_dtype));
  const void** entries = (const void**)malloc(sizeof(void*) * (size_t)W);
  for (uint32_t b = 0; b < batch; ++b) {
    const orc_plan_d* P = &pd[b];
    if (P->seq_len == 0xFFFFFFFFu) continue;
    if (P->write_loc < 0 || (uint64_t)P->write_loc >= state_rows) { free(entries); return ORC_BAD_INDEX; }
    memcpy((char*)state + (size_t)P->write_loc * row_bytes, row_ptr(input, b, width, in_dtype), row_bytes);
    if (P->seq_len % (uint32_t)ratio != 0) continue;
    for (int i = 0; i < W; ++i) {
      if (ratio == 4 && P->seq_len == 4 && i < 4) {
        entries[i] = NULL;
        continue;
      }
      int64_t srow = ratio == 4 ? (int64_t)(i < 4 ? P->read_page_0 : P->read_page_1) * 4 + i % 4
                                : (int64_t)P->read_page_0 * 128 + i;
      if (srow < 0 || (uint64_t)srow >= state_rows) { free(entries); return ORC_BAD_INDEX; }
      entries[i] = row_ptr(state, srow, width, in_dtype);
    }
    pool_window(ratio, hd, in_dtype, out_dtype, (const void* const*)entries, ape,
                (char*)out + (size_t)b * (size_t)hd * elem_size(out_dtype));
  }
  free(entries);
  return ORC_OK;
}

/* The definition with no state at all: given the whole token history of one
 * sequence (rows 0..T-1 in kv_score layout), emit for every position p with
 * (p+1) % ratio == 0 the pool of positions p-W+1 .. p (C4: positions below 0,
 * i.e. the previous group of the first group, are masked).  Token layout:
 * out is [T, hd] with zero rows elsewhere.  Used to pin the prefill / chunked
 * prefill / decode drivers against each other. */
int orc_compress_history(int ratio, int hd, int in_dtype, int out_dtype, const void* tokens, uint32_t T,
                         const void* ape, void* out) {
  int rc = check_common(ratio, hd, in_dtype, out_dtype);
  if (rc) return rc;
  const int W = window_of(ratio);
  const int width = row_width(ratio, hd);
  memset(out, 0, (size_t)T * (size_t)hd * elem_size(out_dtype));
  const void** entries = (const void**)malloc(sizeof(void*) * (size_t)W);
  for (int64_t p = 0; p < (int64_t)T; ++p) {
    if ((p + 1) % ratio != 0) continue;
    for (int i = 0; i < W; ++i) {
      int64_t q = p - (W - 1) + i;
      entries[i] = q < 0 ? NULL : row_ptr(tokens, q, width, in_dtype);
    }
    pool_window(ratio, hd, in_dtype, out_dtype, (const void* const*)entries, ape,
                (char*)out + (size_t)p * (size_t)hd * elem_size(out_dtype));
  }
  free(entries);
  return ORC_OK;
}

/* ----- online C128 state ([cv2] _use_online_compress, generate_online) ---- */

/* The online state pool keeps, per request slot, the running softmax of the
 * current 128-token group instead of the group's 128 rows ([cv2] views the
 * state buffer as [-1, 1, 3 * head_dim] when online compression is on; the
 * online kernels and generate_online themselves are off-page).  Reading: for
 * channel c the slot holds (m, l, a) = (running max of s, sum of exp(s - m),
 * sum of kv * exp(s - m)) over the group's tokens so far; a token at position
 * p with s = fp32(score + ape[p % 128]):
 *   p % 128 == 0:  (m, l, a) <- (s, 1, kv)                       (a new group)
 *   otherwise:     m' = max(m, s);  l <- l e^(m-m') + e^(s-m');
 *                  a <- a e^(m-m') + kv e^(s-m');  m <- m'
 * and when (p + 1) % 128 == 0 the group's row a / l is emitted -- exactly the
 * window softmax of the C128 definition.  The slot of request rid is
 * rid + slot_offset ([cv2] online_state_slot_offset).  The oracle keeps the
 * state in double, [slots, 3 * hd] as (m | l | a). */

typedef struct {
  uint32_t position;   /* first position of the unit */
  uint32_t ragged_cnt; /* ragged id of its first token (24 bits) | token count << 24 (1..128) */
  int32_t slot;
  uint32_t row_flags;  /* compact output row (24 bits) | flags << 24 */
} orc_online_unit;
enum { ORC_UNIT_LOAD = 1, ORC_UNIT_EMIT = 2, ORC_UNIT_STORE = 4 };

/* Prefill units: the tokens of one request inside one 128-group, in the CPU
 * loop order (requests in batch order, positions ascending).  A unit loads the
 * slot when it starts inside a group, emits when it reaches the group's end
 * (its compact output row is the running count of emitting units), and
 * stores the slot when it holds the request's last token. */
int orc_plan_online_prefill(const int64_t* rid, const int64_t* seq_lens, const int64_t* extend_lens, uint32_t batch,
                            uint32_t num_q_tokens, int64_t slot_offset, uint32_t cap_u, int pad_invalid,
                            void* units_out, uint32_t* counts) {
  if (batch > 1024 || num_q_tokens >= (1u << 24)) return ORC_BAD_BATCH;
  orc_online_unit* u = (orc_online_unit*)units_out;
  uint64_t token_base = 0, nu = 0, nc = 0;
  for (uint32_t b = 0; b < batch; ++b) {
    const int64_t sl = seq_lens[b], el = extend_lens[b];
    if (!(0 < el && el <= sl) || sl > INT32_MAX || rid[b] < 0 || rid[b] + slot_offset < 0 ||
        rid[b] + slot_offset > INT32_MAX)
      return ORC_BAD_LENGTH;
    const int64_t pl = sl - el;
    for (int64_t g = pl / 128; g <= (sl - 1) / 128; ++g) {
      const int64_t p0 = pl > 128 * g ? pl : 128 * g;
      const int64_t p1 = sl < 128 * g + 128 ? sl : 128 * g + 128; /* exclusive */
      const int emit = p1 == 128 * g + 128;
      if (nu < cap_u) {
        u[nu].position = (uint32_t)p0;
        u[nu].ragged_cnt = (uint32_t)(token_base + (uint64_t)(p0 - pl)) | ((uint32_t)(p1 - p0) << 24);
        u[nu].slot = (int32_t)(rid[b] + slot_offset);
        const uint32_t flags = (p0 % 128 != 0 ? ORC_UNIT_LOAD : 0) | (emit ? ORC_UNIT_EMIT : 0) |
                               (p1 == sl ? ORC_UNIT_STORE : 0);
        u[nu].row_flags = (uint32_t)(emit ? nc : 0xFFFFFFu) | (flags << 24);
      }
      ++nu;
      nc += emit;
    }
    token_base += (uint64_t)el;
  }
  counts[0] = (uint32_t)nu;
  counts[1] = (uint32_t)nc;
  if (token_base != num_q_tokens) return ORC_BAD_TOTAL;
  if (nu > cap_u) return ORC_CAPACITY;
  if (pad_invalid && cap_u > nu) memset(u + nu, 0xFF, sizeof(orc_online_unit) * (cap_u - nu));
  return ORC_OK;
}

/* One token into channel c's running state (double). */
static void online_step(double* m, double* l, double* a, int first, double s, double kv) {
  if (first) {
    *m = s;
    *l = 1.0;
    *a = kv;
    return;
  }
  const double mn = s > *m ? s : *m;
  const double c = exp(*m - mn), e = exp(s - mn);
  *l = *l * c + e;
  *a = *a * c + kv * e;
  *m = mn;
}

static double online_s(const void* row, int hd, int c, int in_dtype, const void* ape, int64_t p) {
  const float score = load_elem(row, (size_t)hd + c, in_dtype);
  const float bias = load_elem(ape, (size_t)(p % 128) * hd + c, in_dtype);
  return (double)(float)(score + bias); /* one fp32 rounding, as the window form */
}

/* Prefill through the online state: every unit's tokens in order.  Output
 * rows: token layout [num_q_tokens, hd] (an emitted row at the ragged id of
 * its group's last token, every other row +0.0) or compact [out_rows, hd]
 * (row = the unit's output row). */
int orc_online_prefill(int hd, int in_dtype, int out_dtype, double* state, uint64_t slots, const void* input,
                       uint32_t num_q_tokens, const void* ape, const void* units, uint32_t n_units, int out_layout,
                       uint32_t out_rows, void* out) {
  int rc = check_common(128, hd, in_dtype, out_dtype);
  if (rc) return rc;
  const int width = 2 * hd;
  const size_t orow_bytes = (size_t)hd * elem_size(out_dtype);
  if (out_layout == ORC_OUT_TOKEN) memset(out, 0, (size_t)num_q_tokens * orow_bytes);
  const orc_online_unit* u = (const orc_online_unit*)units;
  for (uint32_t k = 0; k < n_units; ++k) {
    if (u[k].position == 0xFFFFFFFFu) continue;
    const uint32_t ragged0 = u[k].ragged_cnt & 0xFFFFFFu, cnt = u[k].ragged_cnt >> 24;
    const uint32_t flags = u[k].row_flags >> 24, orow = u[k].row_flags & 0xFFFFFFu;
    if (u[k].slot < 0 || (uint64_t)u[k].slot >= slots || cnt == 0 || ragged0 + cnt > num_q_tokens)
      return ORC_BAD_INDEX;
    if ((flags & ORC_UNIT_EMIT) && out_layout == ORC_OUT_COMPACT && orow >= out_rows) return ORC_BAD_INDEX;
    double* st = state + (size_t)u[k].slot * 3 * hd;
    for (int c = 0; c < hd; ++c) {
      double m = 0, l = 0, a = 0;
      if (flags & ORC_UNIT_LOAD) {
        m = st[c];
        l = st[hd + c];
        a = st[2 * hd + c];
      }
      for (uint32_t t = 0; t < cnt; ++t) {
        const int64_t p = (int64_t)u[k].position + t;
        const void* row = row_ptr(input, (int64_t)ragged0 + t, width, in_dtype);
        online_step(&m, &l, &a, p % 128 == 0, online_s(row, hd, c, in_dtype, ape, p),
                    (double)load_elem(row, (size_t)c, in_dtype));
      }
      if (flags & ORC_UNIT_STORE) {
        st[c] = m;
        st[hd + c] = l;
        st[2 * hd + c] = a;
      }
      if (flags & ORC_UNIT_EMIT) {
        const size_t r = out_layout == ORC_OUT_TOKEN ? (size_t)(ragged0 + cnt - 1) : (size_t)orow;
        store_elem(out, r * hd + c, out_dtype, a / l);
      }
    }
  }
  return ORC_OK;
}

/* Decode plan for the online state: {seq_len, slot, slot, slot}. */
int orc_plan_online_decode(const int64_t* rid, const int64_t* seq_lens, uint32_t batch, int64_t slot_offset,
                           void* plan_d_out) {
  orc_plan_d* plan = (orc_plan_d*)plan_d_out;
  for (uint32_t b = 0; b < batch; ++b) {
    if (seq_lens[b] < 1 || seq_lens[b] > INT32_MAX || rid[b] < 0 || rid[b] + slot_offset < 0 ||
        rid[b] + slot_offset > INT32_MAX)
      return ORC_BAD_LENGTH;
    const int32_t slot = (int32_t)(rid[b] + slot_offset);
    plan[b].seq_len = (uint32_t)seq_lens[b];
    plan[b].write_loc = slot;
    plan[b].read_page_0 = slot;
    plan[b].read_page_1 = slot;
  }
  return ORC_OK;
}

/* Decode through the online state: row b's token joins slot write_loc; the
 * output is the group's row on a boundary, +0.0 otherwise. */
int orc_online_decode(int hd, int in_dtype, int out_dtype, double* state, uint64_t slots, const void* input,
                      const void* ape, const void* plan_d, uint32_t batch, void* out) {
  int rc = check_common(128, hd, in_dtype, out_dtype);
  if (rc) return rc;
  const int width = 2 * hd;
  memset(out, 0, (size_t)batch * (size_t)hd * elem_size(out_dtype));
  const orc_plan_d* pd = (const orc_plan_d*)plan_d;
  for (uint32_t b = 0; b < batch; ++b) {
    if (pd[b].seq_len == 0xFFFFFFFFu) continue;
    if (pd[b].write_loc < 0 || (uint64_t)pd[b].write_loc >= slots || pd[b].seq_len == 0) return ORC_BAD_INDEX;
    const int64_t p = (int64_t)pd[b].seq_len - 1;
    double* st = state + (size_t)pd[b].write_loc * 3 * hd;
    const void* row = row_ptr(input, b, width, in_dtype);
    for (int c = 0; c < hd; ++c) {
      double m = st[c], l = st[hd + c], a = st[2 * hd + c];
      online_step(&m, &l, &a, p % 128 == 0, online_s(row, hd, c, in_dtype, ape, p),
                  (double)load_elem(row, (size_t)c, in_dtype));
      st[c] = m;
      st[hd + c] = l;
      st[2 * hd + c] = a;
      if ((p + 1) % 128 == 0) store_elem(out, (size_t)b * hd + c, out_dtype, a / l);
    }
  }
  return ORC_OK;
}

/* ----- norm + RoPE + store ([cv2] compress_norm_rope_store step) ---------- */

/* After pooling, each compressed row goes through RMSNorm (weight, eps), then
 * RoPE at position seq_len - ratio (clamped at 0), and is stored into the KV
 * cache at out_loc ([cv2] _forward_compress_all_in_one step 2 and the unified
 * path's steps 2 and 4):
 *   decode  (mode 1): one record per batch row b (a DecodePlan); rows whose
 *                     seq_len is not a multiple of the ratio are zeroed before
 *                     the norm and still stored, at out_loc[b];
 *   prefill (mode 0): one record per CompressPlan entry k; its row is k
 *                     (compact layout) or ragged_id (token layout) and it is
 *                     stored at out_loc[ragged_id].
 * Invalid (all-ones) records are skipped.  RMSNorm: y_c = x_c * w_c /
 * sqrt(mean_c x_c^2 + eps).  RoPE acts on the last rope_dim channels as
 * rope_dim/2 interleaved pairs (2i, 2i+1): (a, b) -> (a cos - b sin,
 * a sin + b cos) with (cos, sin) = freqs[pos][i] (fp32 table, [max_pos,
 * rope_dim/2, 2]).  eps must be positive (the norm of a zeroed row is 0).
 * Everything after reading x is carried in double and rounded once to the
 * cache dtype (RNE). */
int orc_norm_rope_store(int ratio, int mode, int hd, int rope_dim, int in_dtype, const void* rows, int in_layout,
                        uint64_t n_rows, const void* plan, uint32_t n_records, const float* weight, float eps,
                        const float* freqs, uint32_t max_pos, const int64_t* out_loc, uint64_t n_loc,
                        int cache_dtype, void* cache, uint64_t cache_rows) {
  if (ratio != 4 && ratio != 128) return ORC_BAD_RATIO;
  if (hd <= 0 || hd % 128 != 0 || hd > 1024 || rope_dim < 0 || rope_dim % 2 || rope_dim > hd) return ORC_BAD_HEAD_DIM;
  if ((in_dtype != ORC_F32 && in_dtype != ORC_BF16) || (cache_dtype != ORC_F32 && cache_dtype != ORC_BF16))
    return ORC_BAD_DTYPE;
  if (!(eps > 0.0f) || !isfinite(eps)) return ORC_BAD_LENGTH; /* a zero row would give 0 * inf */
  double* y = (double*)malloc(sizeof(double) * (size_t)hd);
  if (!y) return ORC_BAD_BATCH;
  int rc = ORC_OK;
  for (uint32_t k = 0; k < n_records && rc == ORC_OK; ++k) {
    int64_t row, loc_index, pos;
    int zero = 0;
    if (mode == 1) {
      const orc_plan_d* P = (const orc_plan_d*)plan + k;
      if (P->seq_len == 0xFFFFFFFFu) continue;
      row = k;
      loc_index = k;
      zero = P->seq_len % (uint32_t)ratio != 0;
      pos = (int64_t)P->seq_len - ratio;
      if (pos < 0) pos = 0;
    } else {
      const orc_plan_c* P = (const orc_plan_c*)plan + k;
      if (P->seq_len == 0xFFFFFFFFu) continue;
      const int64_t ragged = P->ragged_bl & 0x00FFFFFFu;
      row = in_layout == ORC_OUT_COMPACT ? (int64_t)k : ragged;
      loc_index = ragged;
      pos = (int64_t)P->seq_len - ratio;
    }
    /* the table is read only when there is something to rotate */
    if ((uint64_t)row >= n_rows || (uint64_t)loc_index >= n_loc || pos < 0 ||
        (rope_dim > 0 && pos >= (int64_t)max_pos)) {
      rc = ORC_BAD_INDEX;
      break;
    }
    const int64_t loc = out_loc[loc_index];
    if (loc < 0 || (uint64_t)loc >= cache_rows) {
      rc = ORC_BAD_INDEX;
      break;
    }
    double ss = 0.0;
    for (int c = 0; c < hd; ++c) {
      y[c] = zero ? 0.0 : (double)load_elem(rows, (size_t)row * hd + c, in_dtype);
      ss += y[c] * y[c];
    }
    const double r = 1.0 / sqrt(ss / hd + (double)eps);
    for (int c = 0; c < hd; ++c) y[c] = y[c] * r * (double)weight[c];
    const int base = hd - rope_dim;
    for (int i = 0; i < rope_dim / 2; ++i) {
      const double cs = freqs[((size_t)pos * (rope_dim / 2) + i) * 2];
      const double sn = freqs[((size_t)pos * (rope_dim / 2) + i) * 2 + 1];
      const double a = y[base + 2 * i], b = y[base + 2 * i + 1];
      y[base + 2 * i] = a * cs - b * sn;
      y[base + 2 * i + 1] = a * sn + b * cs;
    }
    for (int c = 0; c < hd; ++c) store_elem(cache, (size_t)loc * hd + c, cache_dtype, y[c]);
  }
  free(y);
  return rc;
}

/* Exposed for the rounding pin (bf16 RNE from a double). */
uint16_t orc_double_to_bf16(double x) { return double_to_bf16_bits(x); }
