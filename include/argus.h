/*
 * argus.h -- C ABI of the GB300 (sm_103a) paged mixed-codec decode-attention library.
 *
 * The operations follow three web pages:
 *   [ARGUS]  "ARGUS: Heterogeneous KV-cache memory management" (argus-cache 0.5.1),
 *            sections "Why decode is slow" and "Direct paged attention".
 *   [PR499]  "feat(kvcache): host-RAM KV tier for sparse-attention models
 *            (--kv-host-pages)" (FreeToken pull request #499) with its update
 *            20f3b23 and the comment describing "--kv-placement host".
 *   [STORE]  "Storage contracts for hybrid KV cache offloading".
 *
 * Conventions shared by every entry point
 *   - Every data pointer is a DEVICE pointer owned by the caller; pointers to
 *     argus_geom / argus_pool / argus_decode_args structs are HOST pointers.
 *   - The library allocates, frees and synchronises nothing.  Every call only
 *     validates its arguments on the host and enqueues kernels on `stream`
 *     (a cudaStream_t; NULL = the legacy default stream).
 *   - The return value reports host-side validation and launch errors only:
 *     ARGUS_E_INVALID for malformed arguments, ARGUS_E_UNSUPPORTED for a
 *     shape / codec combination this build does not implement (there is no
 *     fallback), ARGUS_E_WORKSPACE for a workspace that is too small,
 *     ARGUS_E_LAUNCH when the CUDA launch itself failed.  argus_last_error()
 *     returns a one-line reason for the calling thread's last failure.
 *   - Anomalies found on the device (a block-table slot outside its pool, a
 *     selection entry outside the sequence, more selection entries than the
 *     list width) are never trapped: the kernel skips the entry and adds one
 *     to a caller-provided counter.
 *   - Supported geometry: head_dim in {64, 128}; page_tokens a positive
 *     multiple of 16; n_q_heads a multiple of n_kv_heads with
 *     G = n_q_heads / n_kv_heads between 1 and 8.
 *   - Calls are stateless and thread safe.  Calls that share a workspace
 *     must not run concurrently on the GPU.
 *
 * Pool layout (one pool per codec; a pool is an array of physical page slots):
 *   codes  [n_slots][2 (K, V)][Hkv][P][row]   row = head_dim 16-bit values
 *          (FP16 / BF16), head_dim bytes (FP8 e4m3 / INT8), head_dim/2 bytes
 *          (INT4: two codes per byte, the even element in the low nibble),
 *          head_dim/4 bytes (INT2: element 4k + j in bits 2j, 2j+1 of byte k),
 *          head_dim/8 bytes (INT1: element 8k + j in bit j of byte k)
 *   meta   FP16 / BF16: unused (NULL)
 *          FP8 / INT8:  float [n_slots][2][Hkv]  one scale per (page, head, K|V)
 *          INT4 / INT2 / INT1: half2 {scale, zero} [n_slots][2][Hkv][P][head_dim/32]
 *   Dequantised value: FP8 e4m3_value(code) * scale; INT8 code * scale;
 *   INT4 / INT2 / INT1 code * scale + zero.  INT4 per token and group of 32:
 *   z = fp16_sat(min), s = fp16_sat(RN(RN(max - z) / 15)), code =
 *   clamp(rint(RN(x - z) / s), 0, 15) (s = 0: code 0); INT2 the same with 3
 *   and INT1 with 1 in place of 15.  Codes and pools must be 16-byte aligned.
 */
#ifndef ARGUS_H
#define ARGUS_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  ARGUS_OK = 0,
  ARGUS_E_INVALID = 1,
  ARGUS_E_UNSUPPORTED = 2,
  ARGUS_E_WORKSPACE = 3,
  ARGUS_E_LAUNCH = 4
} argus_status;

/* Codec tiers of [ARGUS] (summary; "Direct paged attention": FP16, Q8, Q4 pages)
 * and [PR499] update 20f3b23 ("e4m3 codes + fp32 scales").  INT2 is the
 * summary's INT2 tier in the "unsigned_affine, bits = 2" form of the ARGUS
 * page's "Pluggable tiers" example, with the INT4 tier's 32-element groups;
 * INT1 is the summary's 1-bit tier in the same form with bits = 1. */
typedef enum {
  ARGUS_FP16 = 0,
  ARGUS_BF16 = 1,
  ARGUS_FP8_E4M3 = 2,
  ARGUS_INT8 = 3,
  ARGUS_INT4_G32 = 4,
  ARGUS_INT2_G32 = 5,
  ARGUS_INT1_G32 = 6
} argus_codec;

typedef struct {
  int32_t n_q_heads;    /* Hq */
  int32_t n_kv_heads;   /* Hkv; G = Hq / Hkv query heads share one KV head */
  int32_t head_dim;     /* D */
  int32_t page_tokens;  /* P */
} argus_geom;

/* Where a pool's pages live ([PR499] "Design" and the comment on
 * "--kv-placement host": a host-RAM tier whose pages attention reads in place).
 * ARGUS_PLACE_HOST: codes and meta are HOST pointers into page-locked memory
 * (cudaHostAlloc / cudaMallocHost / cudaHostRegister) that the device can map;
 * decode reads the selected pages in place over the host link, with plain
 * 16-byte loads, without staging them into device memory.  Accepted by
 * argus_paged_decode_attn (not together with a sliding window or an INT2 pool:
 * ARGUS_E_UNSUPPORTED), argus_paged_window_prefill_attn (staged from host
 * memory) and as the destination of argus_quantize_pages (demotion into the
 * host tier).  Host memory the device cannot map is ARGUS_E_INVALID. */
typedef enum {
  ARGUS_PLACE_DEVICE = 0,
  ARGUS_PLACE_HOST = 1
} argus_placement;

typedef struct {
  int32_t codec;        /* argus_codec of every page in this pool */
  int32_t placement;    /* argus_placement: ARGUS_PLACE_DEVICE (0) or ARGUS_PLACE_HOST */
  void* codes;          /* layout above; device memory, or host memory for ARGUS_PLACE_HOST */
  void* meta;           /* layout above; NULL for FP16 / BF16 */
  int64_t n_slots;      /* physical page slots in the pool */
} argus_pool;

/* ---------------------------------------------------------------------------
 * argus_quantize_pages -- page demotion through the codec tiers.
 *
 * [ARGUS] summary: older pages are demoted from FP16 through FP8, INT8, INT4
 * (and INT2);
 * [PR499] update 20f3b23: the pool holds e4m3 codes + fp32 scales and is the
 * source of truth.  For each listed page i and each (K|V, KV head h) unit:
 *   FP8:  a = max|x| over the unit's valid tokens; scale = a / 448 (fp32);
 *         code = e4m3 round-to-nearest-even, saturating at +-448, of x / scale.
 *   INT8: scale = a / 127; code = clamp(rint_even(x / scale), -127, 127).
 *   INT4: per token and 32-element group: z = fp16_sat(min), s = fp16_sat(
 *         (max - z) / 15); code = s > 0 ? clamp(rint_even((x - z) / s), 0, 15) : 0.
 *   FP16 / BF16 destination (equal to src_dtype): a copy.
 *   a == 0 gives scale 0 and all-zero codes.  Every division is IEEE fp32.
 * Arguments
 *   g            geometry (host)
 *   src_dtype    ARGUS_FP16 or ARGUS_BF16
 *   src_codes    device [n_src_slots][2][Hkv][P][D] 16-bit source pages
 *   src_slots    device int32 [n_pages] source slot of page i
 *   dst          host descriptor of the destination pool
 *   dst_slots    device int32 [n_pages] destination slot of page i
 *   n_pages      pages to demote (0 is a no-op)
 *   valid_tokens device int32 [n_pages] or NULL (= P): tokens >= valid are
 *                left out of the reductions and stored as zero codes / zero meta
 *   ckey_out     device bf16 [n_pages][Hkv][D] or NULL: compressed key of each
 *                page = mean over the valid tokens of the stored (dequantised)
 *                keys, summed in fp32 and rounded to bf16 ([PR499] "Why this
 *                works": the indexer scores a compressed slab)
 * Slots outside their pools are skipped on the device (counted in *status if
 * status != NULL, device uint32).  Source values must be finite: codes for
 * units holding inf or NaN are unspecified.
 * ------------------------------------------------------------------------- */
argus_status argus_quantize_pages(const argus_geom* g, int32_t src_dtype,
                                  const void* src_codes, int64_t n_src_slots,
                                  const int32_t* src_slots, const argus_pool* dst,
                                  const int32_t* dst_slots, int32_t n_pages,
                                  const int32_t* valid_tokens, void* ckey_out,
                                  uint32_t* status, void* stream);

/* ---------------------------------------------------------------------------
 * argus_paged_decode_attn -- single-token decode attention over a paged,
 * mixed-codec KV cache.
 *
 * [ARGUS] "Direct paged attention": an exact tile-by-tile online-softmax
 * recurrence over a structure-of-arrays page table (precision separate from
 * placement); "Why decode is slow": one compressed page at a time, grouped-
 * query attention.  [PR499] "Design": logical pages are translated to physical
 * slots through a block table; "Why this works": attention may be restricted
 * to the indexer's selected pages.  Result, per batch row b and query head hq
 * (KV head h = hq / G):
 *   o = sum_j softmax_j(softmax_scale * q . k_j) v_j,
 *   lse2 = log2 sum_j 2^(softmax_scale * q . k_j * log2 e),
 * over the visible tokens j (positions < seq_lens[b]) of all logical pages, or
 * of the selected pages when sel_pages != NULL; k_j, v_j are dequantised in
 * registers from the page's codec.  An empty visible set gives o = 0 and
 * lse2 = -inf.  Partial results of context splits are folded by log2-sum-exp.
 * ------------------------------------------------------------------------- */
typedef struct {
  argus_geom g;
  int32_t batch;              /* B */
  int32_t q_dtype;            /* ARGUS_FP16 or ARGUS_BF16 */
  const void* q;              /* device [B][Hq][D] */
  const argus_pool* pools;    /* host array, at most one pool per codec */
  int32_t n_pools;
  int32_t max_pages;          /* row length of page_codec / block_table */
  const uint8_t* page_codec;  /* device [B][max_pages] codec of logical page p */
  const int32_t* block_table; /* device [B][max_pages] slot of logical page p */
  const int32_t* seq_lens;    /* device [B] tokens; at most max_pages * P are read */
  const int32_t* sel_pages;   /* device [B][Hkv][sel_width] logical pages, or NULL */
  const int32_t* sel_count;   /* device [B][Hkv] entries used, or NULL */
  int32_t sel_width;
  float softmax_scale;
  void* out;                  /* device [B][Hq][D] in out_dtype (8-byte aligned), or NULL */
  int32_t out_dtype;          /* ARGUS_FP16 or ARGUS_BF16 */
  float* out_f32;             /* device [B][Hq][D] fp32 output (16-byte aligned), or NULL */
  float* lse2_out;            /* device [B][Hq] log2-sum-exp, or NULL */
  uint32_t* status;           /* device uint32 anomaly counter, or NULL */
  int32_t num_splits;         /* context splits per (b, KV head); 0 = automatic.
                                 Dense pages: contiguous chunk ranges.  A selection:
                                 its entries dealt round-robin (split s takes entries
                                 s, s + S, ...), at most sel_width splits */
  int32_t pdl;                /* programmatic dependent launch, see below */
  int32_t window_tokens;      /* > 0: sliding window, see below; 0 = every token */
  int32_t sink_tokens;        /* with a window: leading tokens that stay visible */
} argus_decode_args;

/* Sliding window with sink tokens ([ARGUS] v0.5, "Standalone PageStore /
 * DiskBlockPool": direct attention supports sliding-window masks; the
 * HuggingFace example's sink_tokens = 4).  With window_tokens = W > 0 the
 * decode query of a sequence of L tokens sees the positions p with
 *   L - W <= p < L   or   p < sink_tokens,
 * and nothing else; pages with no visible position are not read.  Dense pages
 * only: W > 0 together with sel_pages is ARGUS_E_UNSUPPORTED; negative values
 * are ARGUS_E_INVALID.  W = 0 ignores sink_tokens.  The workspace and split
 * count are sized for at most ceil(sink/16) + ceil(W/16) + 1 chunks of 16
 * tokens per sequence. */

/* args.status: the decode kernel ORs bit 31 (0x80000000) into *status when
 * one of their waits for a copy or for a sibling warp runs out (2 s).  The
 * results of that call are then undefined; the kernel still ends, and the
 * context stays usable. */

/* args.pdl = 0: the kernels start after their stream predecessor completes
 * (ordinary stream order; always safe).
 * args.pdl = 1: the decode grid may start while its stream predecessor is
 * still running, and it reads page_codec, block_table, seq_lens, sel_pages,
 * sel_count, the pools' codes and meta BEFORE it waits for that predecessor
 * (q is read, and every output written, after the wait).  Set it only when
 * the predecessor does not write those inputs -- for example a previous
 * argus_paged_decode_attn call, layer after layer.  When in doubt, 0.
 * args.pdl = 2: the decode grid may start while its stream predecessor is
 * still running but reads every input after that predecessor completes: always
 * safe, and it hides the launch behind the predecessor's tail (for example
 * after argus_select_pages, which writes sel_pages and sel_count).
 * Other values are ARGUS_E_INVALID. */

/* Workspace needed by argus_paged_decode_attn for these arguments: fp32
 * partial outputs and log2-sum-exp values of the context splits.  Its contents
 * need no initialisation; calls that share a workspace must not overlap on the
 * GPU. */
argus_status argus_decode_workspace_bytes(const argus_decode_args* args, size_t* bytes);

argus_status argus_paged_decode_attn(const argus_decode_args* args, void* ws,
                                     size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * argus_paged_decode_attn_noalloc -- the same decode attention, for callers
 * that cannot allocate device memory.  (The source pages have no counterpart:
 * it is an interface addition of this library.)
 *
 * Who needs it: runtimes whose memory planner hands out all device memory
 * before decoding starts, and host code that may not call cudaMalloc on the
 * decode path (cudaMalloc can synchronise the device).  Such callers cannot
 * provide the workspace argus_paged_decode_attn wants.
 *
 * How it works: the split-combine scratch is a fixed file-scope device array
 * of ARGUS_NOALLOC_SCRATCH_BYTES bytes inside the library; every GPU that
 * loads the library holds it until the process exits.  The caller still
 * passes every input and output in args.  The call allocates nothing: no
 * cudaMalloc, no cudaFree, no allocating library routine.
 *   - The first call on a device resolves the array's device address (with
 *     that device current); make that first call before any stream capture.
 *     The address is resolved again by the first call after the device's
 *     context was destroyed and created anew (cudaDeviceReset), so a stale
 *     address is never used.
 *   - The array keeps the previous call's contents; nothing in it needs to
 *     start at zero (every partial result is written before it is read).
 *   - All calls share the one array: calls that overlap on the GPU (different
 *     streams, or different host threads on the same device) race.  Serialise
 *     them on one stream.
 *   - Arguments whose scratch need (argus_decode_workspace_bytes) exceeds
 *     ARGUS_NOALLOC_SCRATCH_BYTES are rejected with ARGUS_E_WORKSPACE; a
 *     smaller num_splits lowers the need.
 * ------------------------------------------------------------------------- */
#define ARGUS_NOALLOC_SCRATCH_BYTES (4u << 20)

argus_status argus_paged_decode_attn_noalloc(const argus_decode_args* args, void* stream);

/* ---------------------------------------------------------------------------
 * argus_select_pages -- the indexer: top-k page selection over a compressed
 * key slab ([PR499] "Why this works for sparse attention"; "Design": fixed-
 * width list of 2*top_k + 8 entries with a drop counter).
 *   score(b, h, p) = sum over the G query heads of KV head h of q . ckey[b][p][h]
 *   (fp32).  Candidates are pages 0 .. n_pages[b]-1, minus the newest page when
 *   keep_newest; the top_k highest scores are kept (ties to the lower page
 *   index); the newest page is then added.  The list is written in ascending
 *   page order to sel_pages[b][h][0 .. sel_count[b][h]-1]; unused entries are
 *   -1.  Entries that do not fit in sel_width are dropped, lowest score first,
 *   and counted in *drop_counter.
 * Arguments: q device [B][Hq][D] (q_dtype FP16 / BF16); ckeys device bf16
 * [B][max_pages][Hkv][D] in logical page order (q and ckeys 16-byte aligned); n_pages device int32 [B]
 * (values above max_pages are clamped and counted as drops); ws of
 * argus_select_workspace_bytes bytes.  max_pages is at most 65535.
 * The kernels may start while their stream predecessor is still running
 * (programmatic dependent launch); every input is read after it completes
 * (before that, the score grid only prefetches its slab ranges and the
 * queries toward L2, a cache hint that reads nothing into the kernel), and
 * the top-k grid lets its own successor start early in the same way.
 * ------------------------------------------------------------------------- */
argus_status argus_select_workspace_bytes(const argus_geom* g, int32_t batch,
                                          int32_t max_pages, size_t* bytes);

argus_status argus_select_pages(const argus_geom* g, int32_t batch, const void* q,
                                int32_t q_dtype, const void* ckeys,
                                const int32_t* n_pages, int32_t max_pages,
                                int32_t top_k, int32_t keep_newest,
                                int32_t* sel_pages, int32_t* sel_count,
                                int32_t sel_width, uint32_t* drop_counter,
                                void* ws, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * argus_fold_lse -- fold partial attention results into an fp32 accumulator
 * by their log2-sum-exp ([PR499] comment on "--kv-placement host": windows are
 * folded by log2-sum-exp into a float32 accumulator).  In place, per row r:
 *   L = max(La, Lb) + log2(2^(La - max) + 2^(Lb - max));
 *   acc_o = 2^(La - L) acc_o + 2^(Lb - L) part_o;  acc_lse2 = L;
 * a side with lse2 = -inf is the identity.
 * acc_o / part_o device float [n_rows][head_dim]; acc_lse2 / part_lse2 device
 * float [n_rows].  head_dim must be a multiple of 4 and the float arrays
 * 16-byte aligned.
 * ------------------------------------------------------------------------- */
argus_status argus_fold_lse(int64_t n_rows, int32_t head_dim, float* acc_o,
                            float* acc_lse2, const float* part_o,
                            const float* part_lse2, void* stream);

/* ---------------------------------------------------------------------------
 * argus_window_prefill_attn -- attention of a query chunk against one window
 * of cached keys, folded into an fp32 accumulator ([PR499] comment on
 * "--kv-placement host": cached pages are staged into a 131,072-token device
 * window, attended per window, and the windows folded by log2-sum-exp).
 *   Key j of the window is at absolute position win_pos0 + j; query row i at
 *   q_pos0 + i; the key is visible iff win_pos0 + j <= q_pos0 + i.
 *   fold = 0: acc_o / acc_lse2 are overwritten with this window's (o, lse2);
 *   fold = 1: the window's result is folded into them as argus_fold_lse does.
 * Arguments: q device bf16 [Hq][n_q][D]; k, v device bf16 with element
 * (h, j, d) at h * kv_head_stride + j * D + d (kv_head_stride = 0 means
 * win_len * D); acc_o device float [Hq][n_q][D]; acc_lse2 [Hq][n_q].
 * softmax_scale finite and >= 0.  Supported: head_dim 64 or 128, any n_q and
 * win_len (keys past win_len and query rows past n_q are masked).
 * num_splits: key ranges per 128-row query tile, each its own CTA, so that
 * every SM works; their partial results are kept in ws and folded by a second
 * kernel.  1 = one CTA per tile folding directly (ws unused); k > 1 = k ranges;
 * 0 = chosen from the sizes and the SM count when ws != NULL, else 1.
 * ws (device) holds argus_window_prefill_workspace_bytes(..., num_splits)
 * bytes (ARGUS_E_WORKSPACE if smaller); it needs no initialisation, and calls
 * sharing one must not overlap on the GPU.
 * ------------------------------------------------------------------------- */
argus_status argus_window_prefill_workspace_bytes(const argus_geom* g, int32_t n_q,
                                                  int64_t win_len, int32_t num_splits,
                                                  size_t* bytes);

argus_status argus_window_prefill_attn(const argus_geom* g, int32_t n_q,
                                       const void* q, const void* k, const void* v,
                                       int64_t kv_head_stride, int64_t win_len,
                                       int64_t win_pos0, int64_t q_pos0,
                                       float softmax_scale, float* acc_o,
                                       float* acc_lse2, int32_t fold,
                                       int32_t num_splits, void* ws, size_t ws_bytes,
                                       void* stream);

/* ---------------------------------------------------------------------------
 * argus_paged_window_prefill_attn -- the staged prefill over a paged, mixed-
 * codec cache: one window of the cache is staged into device memory through
 * the block table and attended as argus_window_prefill_attn does ([PR499]
 * comment on "--kv-placement host": cached pages are staged into a device
 * window, attended per window, and the windows folded by log2-sum-exp).
 *   The window holds positions win_pos0 .. win_pos0 + win_len - 1 of one
 *   sequence: position p is row p % P of logical page p / P, whose codec and
 *   physical slot are page_codec[p / P] and block_table[p / P] (pages of any
 *   codec, FP8 included).  Key j of the window is at absolute position
 *   win_pos0 + j; query row i at q_pos0 + i; visible iff win_pos0 + j <=
 *   q_pos0 + i.  fold as in argus_window_prefill_attn.
 *   Staging (in the workspace): every key and value of the window is
 *   dequantised from its page's codes and written as fp16, scaled by a power
 *   of two chosen from the window's largest |k| (resp. |v|) so that it lies in
 *   [2^14, 2^15); each query row is written as fp16 scaled the same way by its
 *   own power of two.  Q.K^T and P.V then run in fp16 on the tensor cores with
 *   fp32 accumulation; the powers of two are undone exactly on the scores and
 *   the output.
 * Arguments: q device bf16 [Hq][n_q][D]; pools host array (layout as for
 * argus_paged_decode_attn, at most one pool per codec); page_codec,
 * block_table device [max_pages] rows of the sequence; the window must lie in
 * [0, max_pages * P) (else ARGUS_E_INVALID).  A page whose codec has no pool or
 * whose slot is outside its pool reads as zeros and is counted once per
 * window in *status (device uint32, may be NULL).  ws (device, 16-byte
 * aligned) of argus_paged_window_prefill_workspace_bytes(g, n_q, win_len,
 * num_splits) bytes, required; no initialisation needed.  head_dim 64 or 128.
 * ------------------------------------------------------------------------- */
argus_status argus_paged_window_prefill_workspace_bytes(const argus_geom* g, int32_t n_q,
                                                        int64_t win_len, int32_t num_splits,
                                                        size_t* bytes);

argus_status argus_paged_window_prefill_attn(const argus_geom* g, int32_t n_q, const void* q,
                                             const argus_pool* pools, int32_t n_pools,
                                             const uint8_t* page_codec,
                                             const int32_t* block_table, int32_t max_pages,
                                             int64_t win_pos0, int64_t win_len, int64_t q_pos0,
                                             float softmax_scale, float* acc_o, float* acc_lse2,
                                             int32_t fold, int32_t num_splits, void* ws,
                                             size_t ws_bytes, uint32_t* status, void* stream);

/* ---------------------------------------------------------------------------
 * argus_staging_moves_less -- whether a prefill should stage the cache into
 * device windows (argus_window_prefill_attn) rather than read pages in place.
 *
 * [PR499] comment on "--kv-placement host": when the in-place reads of a
 * prefill's rows add up to more bytes than the cache holds, the cached pages
 * are staged into a device window, attended per window, and the windows
 * folded.  *stage = 1 when
 * the sum of row_read_bytes[0 .. n_rows) is strictly greater than
 * cache_bytes, else 0.
 * Arguments (all HOST memory, no device work): row_read_bytes int64 [n_rows],
 * the bytes each query row would read in place (>= 0); n_rows >= 0;
 * cache_bytes >= 0; stage int32 out.  A NULL pointer (row_read_bytes may be
 * NULL when n_rows = 0) or a negative value is ARGUS_E_INVALID.
 * ------------------------------------------------------------------------- */
argus_status argus_staging_moves_less(const int64_t* row_read_bytes, int64_t n_rows,
                                      int64_t cache_bytes, int32_t* stage);

/* ---------------------------------------------------------------------------
 * Testing only.  argus_test_decode_stall runs argus_paged_decode_attn with
 * every device wait limited to wait_limit_us microseconds (1 .. 2,000,000),
 * and the producer warp (the one issuing copies) of each CTA that reaches stage
 * stall_stage (>= 0; a stage is one ring slot of 16-token chunks) withholds
 * that stage's arrival until the consumer warps have given up on it.  Such a
 * CTA sets bit 31 of *status (args.status is required), waits until every copy
 * it issued has landed, and ends; CTAs with fewer stages run normally.
 * Nothing faults, and each wait ends within wait_limit_us (the producer allows
 * the consumers twice that to give up).  The outputs of the call are
 * undefined.
 * ------------------------------------------------------------------------- */
argus_status argus_test_decode_stall(const argus_decode_args* args, void* ws, size_t ws_bytes,
                                     uint32_t wait_limit_us, int32_t stall_stage, void* stream);

const char* argus_status_string(argus_status s);

/* One-line reason for the calling thread's most recent non-OK status. */
const char* argus_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* ARGUS_H */
