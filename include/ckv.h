/*
 * ckv.h -- C ABI of libckv, the GB300 (sm_103a) KV compressor for
 * DeepSeek-V4-style compressed attention caches.
 *
 * What it computes.  Every request owns a small state buffer: an 8-slot ring
 * for compress ratio 4 ("C4") and a 128-slot page for ratio 128 ("C128").
 * Each new token contributes one kv_score row:
 *     C4   row = | kv-overlap | kv | score-overlap | score |   (4 * head_dim)
 *     C128 row = | kv | score |                               (2 * head_dim)
 * Whenever a request's length reaches a multiple of the ratio, one compressed
 * KV row of head_dim values is emitted: per channel c, a softmax over the
 * window of (score + ape[i]) weights the kv values,
 *     out[c] = sum_i kv_i[c] * exp(s_i[c] - m) / sum_i exp(s_i[c] - m),
 *     s_i[c] = fp32(score_i[c]) + fp32(ape[i][c]),  m = max_i s_i[c].
 * C4's window is 8 tokens: the previous group's 4 overlap halves followed by
 * the current group's 4 main halves; for the first group (length 4) the
 * previous group does not exist and is left out.  C128's window is the 128
 * tokens of the page.
 *
 * Sources (SGLang DeepSeek-V4 compressor): c_plan.cuh (the CompressPlan /
 * WritePlan / DecodePlan builders and the legacy ring/page addressing),
 * c4.cuh (C4 write and pool: c4_write, c4_forward, flash_c4_decode,
 * flash_c4_prefill, FlashCompress4Kernel::run_prefill launch order),
 * compressor_v2.py (C128 write and pool: _c128_compress_decode_kernel,
 * _c128_compress_prefill_write_kernel, _compress_forward_c128_fallback).
 *
 * Conventions for every entry point:
 *  - All pointers are DEVICE pointers owned by the caller (for example PyTorch
 *    allocations).  The library allocates no device or host memory.
 *  - Work is enqueued on `stream` and the call returns without synchronising;
 *    results are valid once the stream has reached that point.  No call reads
 *    device data on the host, so every call can be captured in a CUDA graph.
 *  - The return value reports argument errors found on the host (CKV_OK or a
 *    negative CKV_ERR_* code; nothing is launched on error).  Problems found in
 *    device-resident data (bad lengths, out-of-range indices) are OR-ed into
 *    the caller's `d_status` word (a device uint32, CKV_STATUS_* bits; may be
 *    NULL to ignore them); the affected records are skipped, never trapped on.
 *  - Pointers must be 16-byte aligned; head_dim must be a multiple of 128 and
 *    at most 1024; dtypes are CKV_F32 or CKV_BF16.
 *  - State buffers: C4 state is [num_requests * 8, 4 * head_dim] (request rid
 *    owns rows rid*8 .. rid*8+7, i.e. two 4-slot pages 2*rid and 2*rid+1);
 *    C128 state is [num_requests * 128, 2 * head_dim] (page rid = rows
 *    rid*128 .. rid*128+127).  The state dtype is the input dtype.
 *  - Invalid plan records have every byte 0xFF and are skipped.
 */
#ifndef CKV_H_
#define CKV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* ckv_stream_t; /* the same handle as cudaStream_t */

/* ------------------------------------------------------------------ codes */
enum { CKV_F32 = 0, CKV_BF16 = 1 };
enum { CKV_OUT_TOKEN = 0, CKV_OUT_COMPACT = 1 };

enum {
  CKV_OK = 0,
  CKV_ERR_RATIO = -1,    /* ratio is not 4 or 128 */
  CKV_ERR_HEAD_DIM = -2, /* head_dim not a positive multiple of 128, or > 1024 */
  CKV_ERR_SIZE = -3,     /* batch > 1024, num_q_tokens >= 2^24, or a size/capacity out of range */
  CKV_ERR_POINTER = -4,  /* a required pointer is NULL or not 16-byte aligned */
  CKV_ERR_DTYPE = -5,    /* unsupported dtype / layout code */
  CKV_ERR_LAUNCH = -6    /* the CUDA launch failed (cudaGetLastError) */
};

/* Bits OR-ed into *d_status by device code. */
enum {
  CKV_STATUS_BAD_LENGTH = 1u,  /* a request with extend_len <= 0, extend_len > seq_len,
                                  seq_len >= 2^31, or a negative / too large rid */
  CKV_STATUS_BAD_TOTAL = 2u,   /* sum(extend_lens) != num_q_tokens */
  CKV_STATUS_CAPACITY = 4u,    /* more plan records than capacity_c / capacity_w */
  CKV_STATUS_BAD_INDEX = 8u,   /* a plan record points outside the state or the input */
  CKV_STATUS_TIMEOUT = 16u     /* a bounded wait on an asynchronous copy expired */
};

enum { CKV_MAX_BATCH = 1024, CKV_MAX_TOKENS = (1 << 24) - 1 };

/* ------------------------------------------------------------------ waits */
/* The pooling kernels that stage their inputs through the TMA engine (C4 and
 * C128 prefill pools, C128 decode, online prefill) wait on mbarriers for those
 * copies (small C4 prefill steps, which load their windows directly, have no
 * such waits).  Every such wait gives up after a time limit: the kernel then ORs
 * CKV_STATUS_TIMEOUT into *d_status and its CTA stops, after waiting (up to
 * 2 s) for the copies it has already issued, so that none of them lands in
 * shared memory the CTA no longer owns.  The context stays usable.
 *
 * ckv_set_wait_limit_ns sets that limit, in nanoseconds, for every launch made
 * after the call, process-wide (an atomic; calls from several threads are
 * safe), and returns the previous limit.  0 restores the default, 2 s; limits
 * above 10 s are clamped to 10 s, so that every wait stays bounded.  A
 * launch captured in a CUDA graph keeps the limit in force at its capture.  The
 * outputs of a launch whose waits expired -- and, for a decode, the state row
 * it writes -- are unspecified; a limit below a copy's latency (a few
 * microseconds) makes the waits expire on purpose.  Host only: touches no
 * device and cannot fail. */
uint64_t ckv_set_wait_limit_ns(uint64_t limit_ns);

/* ------------------------------------------------------------------ plans */
/* One compress event (16 bytes).  seq_len = position + 1 (a multiple of the
 * ratio); ragged_bl = ragged_id | buffer_len << 24 where ragged_id is the row of
 * the event's own token in the ragged input and buffer_len is the number of
 * leading window entries held in the state (the rest are ragged rows
 * ragged_id - (W-1) + i); read_page_0 / read_page_1 are the state pages of
 * position max(position - ratio, 0) and of position (C4: 4-slot pages, window
 * entries 0..3 live in read_page_0, entries 4..7 in read_page_1, slot i % 4;
 * C128: page read_page_0, slot i).  c_plan.cuh: plan_compress_prefill (the
 * CPU loop) and plan_compress_prefill_legacy_kernel; ragged_id widened from 16
 * to 24 bits. */
typedef struct ckv_compress_plan {
  uint32_t seq_len;
  uint32_t ragged_bl;
  int32_t read_page_0;
  int32_t read_page_1;
} ckv_compress_plan_t;

/* One state write (8 bytes): state[write_loc] = input[ragged_id].
 * c_plan.cuh: WritePlan after plan_compress_prefill_legacy_kernel. */
typedef struct ckv_write_plan {
  uint32_t ragged_id;
  int32_t write_loc;
} ckv_write_plan_t;

/* One decode row (16 bytes): seq_len, the state row the new token goes to, and
 * the pages of positions max(seq_len-1-ratio, 0) and seq_len-1.
 * c_plan.cuh: plan_compress_decode_legacy_kernel. */
typedef struct ckv_decode_plan {
  uint32_t seq_len;
  int32_t write_loc;
  int32_t read_page_0;
  int32_t read_page_1;
} ckv_decode_plan_t;

/* The page-boundary rows of a decode batch, in row order (8 bytes per
 * entry; written by ckv_plan_decode / ckv_plan_decode_paged when asked for,
 * read by ckv_compress_decode).  An array of batch + 1 entries: entry 0 is
 * {count, 0}, entries 1 .. count are {row, read_page_0} of the rows whose
 * record is valid and whose seq_len is a multiple of the ratio (the rows that
 * emit a compressed row); entries past count are not written.  The pages
 * define no such list: it lets the C128 decode hand out its windows to the
 * SMs without every CTA scanning the whole plan first. */
typedef struct ckv_decode_order {
  uint32_t row;
  int32_t page;
} ckv_decode_order_t;

/* Prefetch hints for the prefill pool (32 bytes, host memory): the device
 * arrays [batch] that ckv_plan_prefill read for this step (int64, 8-byte
 * aligned; all three or none).  The pages define no such thing: the pool
 * reads them BEFORE waiting for the previous kernel on the stream (normally
 * the planner), only to prefetch into L2 the state rows of the windows they
 * imply while that kernel runs (legacy rows: ring rid * 8 + position % 8 for
 * C4, page rid * 128 + position % 128 for C128).  Nothing is computed from
 * them: a stale or wrong value costs the bandwidth of a useless prefetch,
 * rows outside the state are skipped, and with SWA-paged plans the prefetch
 * simply misses.  The pool uses them only for small steps (input of at most
 * CKV_PREFILL_HINT_MAX_INPUT_BYTES), where the windows' first loads, not the
 * stream of windows, set the time. */
typedef struct ckv_prefill_hints {
  const int64_t* rid;
  const int64_t* seq_lens;
  const int64_t* extend_lens;
  uint32_t batch;
  uint32_t reserved; /* 0 */
} ckv_prefill_hints_t;

#define CKV_PREFILL_HINT_MAX_INPUT_BYTES (64ull << 20)

#define CKV_RAGGED_MASK 0x00FFFFFFu
#define CKV_BUFFER_LEN_SHIFT 24

/* One online-state prefill unit (16 bytes): the tokens of one request that
 * fall inside one 128-group (see "Online C128 state" below).  Invalid = all
 * bytes 0xFF. */
typedef struct ckv_online_unit {
  uint32_t position;   /* position of the unit's first token */
  uint32_t ragged_cnt; /* ragged id of that token (24 bits) | token count (1..128) << 24 */
  int32_t slot;        /* the request's state slot */
  uint32_t row_flags;  /* compact output row (24 bits, all ones when nothing is emitted) | flags << 24 */
} ckv_online_unit_t;

#define CKV_UNIT_COUNT_SHIFT 24
#define CKV_UNIT_FLAGS_SHIFT 24
enum {
  CKV_UNIT_LOAD = 1u,  /* the unit starts inside a group: continue from the slot */
  CKV_UNIT_EMIT = 2u,  /* the unit ends its group: emit the group's row */
  CKV_UNIT_STORE = 4u  /* the unit holds the request's last token: store the slot */
};

/* Upper bounds a caller can size plan buffers with (host arithmetic only):
 * compress records <= num_q_tokens / ratio + batch, and
 * write records <= min(num_q_tokens, batch * (ratio == 4 ? 7 : 127)). */
uint32_t ckv_capacity_compress(int ratio, uint32_t batch, uint32_t num_q_tokens);
uint32_t ckv_capacity_write(int ratio, uint32_t batch, uint32_t num_q_tokens);

/* Decode plan (c_plan.cuh plan_compress_decode_legacy_kernel).
 * rid[batch], seq_lens[batch]: int64 device arrays (seq_len counts the new
 * token).  plan_d[batch]: output.  Rows with bad values get an invalid record
 * and set CKV_STATUS_BAD_LENGTH.  order: NULL, or an 8-byte aligned output
 * of batch + 1 ckv_decode_order_t entries that receives the batch's
 * page-boundary rows (see ckv_decode_order_t).  Without order: one launch of
 * ceil(batch/256) x 256 threads; with order: one CTA of 1024 threads (a
 * block-wide scan of the batch, so the list comes out in row order). */
int ckv_plan_decode(int ratio, const int64_t* rid, const int64_t* seq_lens, uint32_t batch,
                    ckv_decode_plan_t* plan_d, ckv_decode_order_t* order, uint32_t* d_status, ckv_stream_t stream);

/* Prefill plans (c_plan.cuh plan_compress_prefill_kernel0 / _kernel_1 and the
 * CPU loop of plan_compress_prefill_legacy, whose order is reproduced exactly):
 * requests in batch order, positions ascending; compress records and write
 * records are separate lists.  A request b with prefix pl = seq_lens[b] -
 * extend_lens[b] emits a compress record for every extend position p with
 * (p+1) % ratio == 0 and a write record for every extend position
 * p >= (seq_len/ratio)*ratio - (ratio == 4 ? 4 : 0).
 * Inputs: rid, seq_lens, extend_lens int64 device arrays [batch], batch <= 1024,
 * num_q_tokens = sum(extend_lens) < 2^24 (checked on the device).
 * Outputs: plan_c[capacity_c], plan_w[capacity_w]; d_counts[4] = {num_c, num_w,
 * min extend_len, max extend_len} (num_c / num_w are the true counts even when
 * they exceed the capacity; records past the capacity are dropped and
 * CKV_STATUS_CAPACITY is set).  With pad_invalid != 0 the records
 * [count, capacity) are filled with the invalid record (fixed-shape buffers for
 * CUDA graphs).  One launch: every CTA scans the <= 1024 lengths itself and then
 * emits its share of records, so no workspace is needed. */
int ckv_plan_prefill(int ratio, const int64_t* rid, const int64_t* seq_lens, const int64_t* extend_lens,
                     uint32_t batch, uint32_t num_q_tokens, uint32_t capacity_c, uint32_t capacity_w,
                     int pad_invalid, ckv_compress_plan_t* plan_c, ckv_write_plan_t* plan_w, uint32_t* d_counts,
                     uint32_t* d_status, ckv_stream_t stream);

/* SWA-paged planners (c_plan.cuh plan_compress_prefill / plan_compress_decode
 * with plan_compress_prefill_kernel_1 / plan_compress_decode_kernel: the main,
 * non-legacy path of that page).
 * C4: state rows come from the request's token map.  For position p of
 * request rid, full = req_to_token[rid * r2t_stride + p] (int32), swa =
 * full_to_state[full] (int64), and the row is
 *     (swa / swa_page_size) * ring_size + swa % ring_size,
 * i.e. every SWA page owns a ring of ring_size rows; read pages are rows / 4.
 * The write set adds, to the legacy one, the last 4 positions of every SWA
 * page in the extend (the next page's first window reads them as its previous
 * group), and keeps positions >= seq_len - mtp_pad with mtp_pad =
 * min(ring_size - ratio, 4) (the GPU-input planner's rule; with the rings
 * accepted here it adds nothing).  Requirements: swa_page_size % ring_size ==
 * 0, ring_size % 4 == 0, ring_size >= 8 (a 4-row ring would put a window's two
 * groups in one page); the pooling kernels assume that the 4 positions of a
 * group sit in the 4 slots of one 4-slot page, true for any page-granular SWA
 * allocation.  A request with rid >= num_reqs or seq_len > r2t_stride, or a
 * mapping entry out of range or negative, yields invalid records and
 * CKV_STATUS_BAD_INDEX (device-side).
 * C128: state is request-scoped (rid * ring_size + p % ring_size) and the maps
 * are not read (they may be NULL).  ring_size must be 128: the C128 pooling
 * reads its window from read_page_0, which is the window's own page only for a
 * 128-row ring.  Decode plans and write records are then the legacy ones.
 * Prefill compress records with buffer_len == 0 read no state; as kernel_1
 * leaves them, their read_page_0 is -1 and read_page_1 the request's index in
 * the batch (both ratios).  Capacities: compress records as
 * ckv_capacity_compress, write records <= ckv_capacity_write_paged. */
uint32_t ckv_capacity_write_paged(int ratio, uint32_t batch, uint32_t num_q_tokens, int32_t swa_page_size);

int ckv_plan_prefill_paged(int ratio, const int64_t* rid, const int32_t* req_to_token, int64_t r2t_stride,
                           uint32_t num_reqs, const int64_t* full_to_state, uint64_t num_full_slots,
                           int32_t swa_page_size, int32_t ring_size, const int64_t* seq_lens,
                           const int64_t* extend_lens, uint32_t batch, uint32_t num_q_tokens, uint32_t capacity_c,
                           uint32_t capacity_w, int pad_invalid, ckv_compress_plan_t* plan_c,
                           ckv_write_plan_t* plan_w, uint32_t* d_counts, uint32_t* d_status, ckv_stream_t stream);

int ckv_plan_decode_paged(int ratio, const int64_t* rid, const int32_t* req_to_token, int64_t r2t_stride,
                          uint32_t num_reqs, const int64_t* full_to_state, uint64_t num_full_slots,
                          int32_t swa_page_size, int32_t ring_size, const int64_t* seq_lens, uint32_t batch,
                          ckv_decode_plan_t* plan_d, ckv_decode_order_t* order, uint32_t* d_status,
                          ckv_stream_t stream);

/* ------------------------------------------------------------------ compute */
/* Prefill state write (c4.cuh c4_write / flash_c4_prefill<kWrite=true>,
 * compressor_v2.py _c128_compress_prefill_write_kernel): for each of the first
 * min(d_counts[1], capacity_w) records (all capacity_w records when d_counts is
 * NULL), copy input row ragged_id (width 4*hd for C4, 2*hd for C128) to state
 * row write_loc, bit for bit.  state_rows = rows of the state buffer.  Must run
 * after ckv_compress_pool_prefill of the same step (writes may overwrite slots
 * that the step's windows still read). */
int ckv_compress_write(int ratio, int head_dim, int dtype, void* state, uint64_t state_rows,
                       const void* kv_score_input, uint32_t num_q_tokens, const ckv_write_plan_t* plan_w,
                       const uint32_t* d_counts, uint32_t capacity_w, uint32_t* d_status, ckv_stream_t stream);

/* Prefill pool (c4.cuh c4_forward via flash_c4_prefill<kWrite=false>;
 * compressor_v2.py _compress_forward_c128_fallback): for each compress record
 * (the first min(d_counts[0], capacity_c)), window entry i < buffer_len is read
 * from the state, the rest from input rows ragged_id - (W-1) + i; C4 records
 * with seq_len == 4 leave out entries 0..3.  Output, in out_dtype:
 *   CKV_OUT_TOKEN:   out is [num_q_tokens, head_dim]; row ragged_id holds the
 *                    compressed row, every other row is written with +0.0.
 *   CKV_OUT_COMPACT: out is [capacity_c, head_dim]; row k holds record k
 *                    (rows of invalid / missing records are left untouched).
 * ape is [W, head_dim] in the input dtype (W = 8 or 128).  Only reads the state.
 * hints: NULL, or ckv_prefill_hints_t (see there); CKV_ERR_POINTER when its
 * arrays are not all given or not 8-byte aligned. */
int ckv_compress_pool_prefill(int ratio, int head_dim, int in_dtype, int out_dtype, const void* state,
                              uint64_t state_rows, const void* kv_score_input, uint32_t num_q_tokens,
                              const void* ape, const ckv_compress_plan_t* plan_c, const uint32_t* d_counts,
                              uint32_t capacity_c, int out_layout, void* out, const ckv_prefill_hints_t* hints,
                              uint32_t* d_status, ckv_stream_t stream);

/* Prefill step: ckv_compress_pool_prefill followed by ckv_compress_write on
 * the same stream (the order of c4.cuh FlashCompress4Kernel::run_prefill). */
int ckv_compress_prefill(int ratio, int head_dim, int in_dtype, int out_dtype, void* state, uint64_t state_rows,
                         const void* kv_score_input, uint32_t num_q_tokens, const void* ape,
                         const ckv_compress_plan_t* plan_c, const ckv_write_plan_t* plan_w,
                         const uint32_t* d_counts, uint32_t capacity_c, uint32_t capacity_w, int out_layout,
                         void* out, const ckv_prefill_hints_t* hints, uint32_t* d_status, ckv_stream_t stream);

/* Decode (c4.cuh flash_c4_decode; compressor_v2.py _c128_compress_decode_kernel):
 * for each row b, write input row b to state row plan_d[b].write_loc; when
 * seq_len % ratio == 0 emit the pool of the window (the new token's entry is
 * taken from the input row, the others from the state), otherwise write +0.0
 * to out row b.  kv_score_input is [batch, width], out is [batch, head_dim].
 * Two rows of one batch must not name the same request.
 * order: NULL, or the list that ckv_plan_decode wrote next to plan_d (8-byte
 * aligned, batch + 1 entries).  The C128 decode then reads only its own
 * entries of the list instead of scanning the plan for the rows that emit;
 * the C4 decode does not read it.  A list that does not match plan_d is a
 * caller error: its entries are still bounds-checked (a row >= batch or a
 * page outside the state is skipped with CKV_STATUS_BAD_INDEX), but the
 * outputs are then unspecified.
 * rid_hint, seq_lens_hint: NULL, or the int64 arrays [batch] the decode
 * planner read (8-byte aligned; both or neither).  The C128 decode reads them
 * BEFORE waiting for the previous kernel on the stream, only to prefetch the
 * windows of page-boundary rows (page = rid, as both C128 decode planners
 * give it) into L2 while that kernel finishes; nothing is computed from them.
 * If the previous kernel is still writing them, a stale value only costs
 * the bandwidth of a useless prefetch; pages outside the state are skipped.
 * The C4 decode likewise prefetches the ring rows its windows read, assuming
 * the legacy ring (rows rid * 8 .. rid * 8 + 7; with SWA-paged plans the
 * prefetch misses and only costs bandwidth). */
int ckv_compress_decode(int ratio, int head_dim, int in_dtype, int out_dtype, void* state, uint64_t state_rows,
                        const void* kv_score_input, const void* ape, const ckv_decode_plan_t* plan_d,
                        const ckv_decode_order_t* order, const int64_t* rid_hint, const int64_t* seq_lens_hint,
                        uint32_t batch, void* out, uint32_t* d_status, ckv_stream_t stream);

/* ------------------------------------------------------- online C128 state */
/* compressor_v2.py can keep C128 state online: one slot of 3 * head_dim per
 * request ([slots, 1, 3 * head_dim]) instead of a 128-row page; the online
 * kernels and their plans (generate_online) are off-page, so this is a
 * derivation.  Slot layout, fp32: m2 | l | a, each head_dim wide: per
 * channel, over the tokens of the current 128-group so far, with m the running
 * maximum of s = fp32(score + ape[p % 128]): m2 = fp32(m * log2(e)),
 * l = sum exp(s - m) and a = sum kv exp(s - m).
 * A token at position p starts a new group when p % 128 == 0 ((m, l, a) =
 * (s, 1, kv)) and otherwise folds in, rescaling by exp(m_old - m_new) when it
 * raises the maximum; at (p + 1) % 128 == 0 the group's row a / l is emitted,
 * which is the C128 window softmax.  The slot of request rid is
 * rid + slot_offset (compressor_v2.py online_state_slot_offset).
 *
 * Prefill: ckv_plan_online_prefill emits one unit per (request, group that
 * the request's extend touches), in batch order and position order, into
 * units[capacity_u] (<= ckv_capacity_online_units); d_counts receives
 * {num_c (units that emit), num_units, min extend_len, max extend_len}; the
 * length checks, status bits and pad_invalid are those of ckv_plan_prefill.
 * An emitting unit's compact output row is its rank among emitting units,
 * i.e. the compress record order of the legacy planner. */
uint32_t ckv_capacity_online_units(uint32_t batch, uint32_t num_q_tokens);

int ckv_plan_online_prefill(const int64_t* rid, const int64_t* seq_lens, const int64_t* extend_lens,
                            uint32_t batch, uint32_t num_q_tokens, int64_t slot_offset, uint32_t capacity_u,
                            int pad_invalid, ckv_online_unit_t* units, uint32_t* d_counts, uint32_t* d_status,
                            ckv_stream_t stream);

/* Runs the first min(d_counts[1], capacity_u) units (all when d_counts is NULL)
 * through the state (fp32 [slots, 3 * head_dim], read and written).  Outputs:
 * CKV_OUT_TOKEN: out [num_q_tokens, head_dim], an emitted row at the ragged id
 * of its group's last token and +0.0 in every other row the units cover;
 * CKV_OUT_COMPACT: out [out_rows, head_dim], row = the unit's output row.
 * Units naming a slot >= slots, rows past num_q_tokens or an output row >=
 * out_rows are skipped with CKV_STATUS_BAD_INDEX.  Units of different
 * requests must name different slots; the units of one request share its
 * slot, and the library reads the slot for the request's first unit before
 * any unit of the call stores it (two launches: the second one stores the
 * state of last units that start at a group start). */
int ckv_compress_online_prefill(int head_dim, int in_dtype, int out_dtype, float* state, uint64_t slots,
                                const void* kv_score_input, uint32_t num_q_tokens, const void* ape,
                                const ckv_online_unit_t* units, const uint32_t* d_counts, uint32_t capacity_u,
                                int out_layout, uint32_t out_rows, void* out, uint32_t* d_status,
                                ckv_stream_t stream);

/* Decode: plan record b = {seq_len, slot, slot, slot} (slot = rid + slot_offset);
 * the compute folds row b of kv_score_input [batch, 2 * head_dim] into its
 * slot and writes out row b: the group's row when seq_len % 128 == 0, +0.0
 * otherwise.  Two rows of one batch must not name the same slot. */
int ckv_plan_online_decode(const int64_t* rid, const int64_t* seq_lens, uint32_t batch, int64_t slot_offset,
                           ckv_decode_plan_t* plan_d, uint32_t* d_status, ckv_stream_t stream);

int ckv_compress_online_decode(int head_dim, int in_dtype, int out_dtype, float* state, uint64_t slots,
                               const void* kv_score_input, const void* ape, const ckv_decode_plan_t* plan_d,
                               uint32_t batch, void* out, uint32_t* d_status, ckv_stream_t stream);

/* ------------------------------------------------------- norm, RoPE, store */
/* The step after pooling (compressor_v2.py compress_norm_rope_store and the
 * unified path's steps 2-4): every compressed row is normalised, rotated and
 * stored into the KV cache.
 *   y_c = x_c * norm_weight[c] / sqrt(mean_c(x_c^2) + eps)        (RMSNorm)
 * then the last rope_dim channels turn as interleaved pairs (2i, 2i+1):
 *   (a, b) -> (a*cos - b*sin, a*sin + b*cos),  (cos, sin) = freqs[pos][i],
 * with pos = max(seq_len - ratio, 0) from the row's plan record, and y is
 * written, rounded to cache_dtype, to kv_cache row out_loc.
 *   rows       the pooled output (in_dtype CKV_F32 or CKV_BF16).
 *   norm_weight fp32 [head_dim]; eps > 0 (else CKV_ERR_SIZE).
 *   freqs      fp32 [max_pos, rope_dim/2, 2] (cos, sin); rope_dim a multiple
 *              of 4, 0 <= rope_dim <= head_dim (else CKV_ERR_HEAD_DIM).  The
 *              table and the channel split are the caller's (compressor_v2.py
 *              takes both from the model).  With rope_dim 0 the table is
 *              not read (freqs may be NULL).
 *   kv_cache   [cache_rows, head_dim] of cache_dtype (CKV_BF16 or CKV_F32).
 * Records whose position, row or out_loc falls outside the table, the rows
 * or the cache are skipped with CKV_STATUS_BAD_INDEX.  Runs after the pooling
 * of the same step on the same stream.
 *
 * Prefill: one record per CompressPlan entry (the first min(d_counts[0],
 * capacity_c); all capacity_c when d_counts is NULL; invalid ones skipped).
 * Its row is k (in_layout CKV_OUT_COMPACT) or ragged_id (CKV_OUT_TOKEN) of
 * rows [n_rows, head_dim]; it is stored at out_loc[ragged_id] (out_loc is
 * int64 [n_out_loc], indexed by token). */
int ckv_norm_rope_store_prefill(int ratio, int head_dim, int rope_dim, int in_dtype, const void* rows,
                                int in_layout, uint64_t n_rows, const ckv_compress_plan_t* plan_c,
                                const uint32_t* d_counts, uint32_t capacity_c, const float* norm_weight, float eps,
                                const float* freqs, uint32_t max_pos, const int64_t* out_loc, uint64_t n_out_loc,
                                int cache_dtype, void* kv_cache, uint64_t cache_rows, uint32_t* d_status,
                                ckv_stream_t stream);

/* Decode: row b of rows [batch, head_dim] with DecodePlan record b; rows whose
 * seq_len is not a multiple of the ratio are zeroed before the norm and are
 * still stored, at out_loc[b] (int64 [batch]), as compressor_v2.py does with
 * its dummy location 0. */
int ckv_norm_rope_store_decode(int ratio, int head_dim, int rope_dim, int in_dtype, const void* rows,
                               const ckv_decode_plan_t* plan_d, uint32_t batch, const float* norm_weight, float eps,
                               const float* freqs, uint32_t max_pos, const int64_t* out_loc, int cache_dtype,
                               void* kv_cache, uint64_t cache_rows, uint32_t* d_status, ckv_stream_t stream);

/* Decode with norm + RoPE + store in one launch, ratio 4 only (the step that
 * compressor_v2.py runs after the C4 decode, fused; the pages run them as two
 * steps): exactly ckv_compress_decode with an fp32 output followed by
 * ckv_norm_rope_store_decode on that output -- the state write, the pooled
 * row (or +0.0 off a group boundary) normalised, rotated at table row
 * max(seq_len - 4, 0) and stored at kv_cache row out_loc[b] -- except that the
 * pooled rows are never written to memory, and the RMS's fp32 sum of squares
 * runs in another order (results agree within the norm step's rounding).  A
 * row's 4-channel units are threads of one block, so the norm needs no second
 * launch; the C128 decode spreads a row over several CTAs and has no such
 * form (CKV_ERR_RATIO).  Arguments as in ckv_compress_decode (without order and
 * out) and ckv_norm_rope_store_decode (without rows and in_dtype); out_loc is
 * int64 [batch].  Invalid records store nothing; a row whose record points
 * outside the state is flagged CKV_STATUS_BAD_INDEX, writes no state and stores
 * the normalised zero row; a position outside the table or a location outside
 * the cache is flagged and stores nothing. */
int ckv_compress_decode_norm_rope_store(int ratio, int head_dim, int rope_dim, int in_dtype, void* state,
                                        uint64_t state_rows, const void* kv_score_input, const void* ape,
                                        const ckv_decode_plan_t* plan_d, const int64_t* rid_hint,
                                        const int64_t* seq_lens_hint, uint32_t batch, const float* norm_weight,
                                        float eps, const float* freqs, uint32_t max_pos, const int64_t* out_loc,
                                        int cache_dtype, void* kv_cache, uint64_t cache_rows, uint32_t* d_status,
                                        ckv_stream_t stream);

/* ------------------------------------------------------------------ misc */
/* Short text for a CKV_OK / CKV_ERR_* code (static storage). */
const char* ckv_error_string(int code);
/* Library ABI version: major * 100 + minor (220: 2.00's decode boundary-row
 * list and prefetch hints, 2.10's prefill prefetch hints, and the fused C4
 * decode + norm + RoPE + store). */
int ckv_version(void);

#ifdef __cplusplus
}
#endif

#endif /* CKV_H_ */
