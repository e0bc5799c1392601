// argus_select_pages: the sparse-attention indexer -- top-k page selection
// over a compressed-key slab.
//
// "feat(kvcache): host-RAM KV tier for sparse-attention models", section "Why
// this works for sparse attention": every attend step first runs top-k block
// selection over a compressed slab, GPU resident and fixed shape, then reads
// only the selected pages; section "Design": the selection is compacted into a
// fixed-width list of 2*block_topk + 8 entries with a drop counter instead of
// silent corruption.
//   score(b, h, p) = sum over the G query heads of KV head h of q . ckey[b][p][h]
//   candidates 0 .. n-2 (n-1 when keep_newest is off); top_k by score, ties to
//   the lower page index; the newest page is always added; ascending order.
//
// GB300 design: two launches.  (1) score: the slab is the dominant HBM stream
// (D bf16 per page and head); one wave of CTAs tiles (batch row, page range).
// A CTA prefetches its range toward L2 before waiting for its stream
// predecessor, then streams it into shared memory with bulk copies; lanes
// read 16 bytes of a compressed key each and fold eight rows' partial dot
// products across the head's lanes in one transposed reduction; the G-query
// sum is formed once per CTA and kept in registers; scores are stored as
// order-preserving uint32 keys.  Each CTA also reports, per KV head, the 2
// largest keys of its own page range.
// (2) top-k: one CTA per (batch row, KV head).  The row's k-th largest key T is
// at least the k-th largest of the reported keys (they are keys of distinct
// pages of the row), and since the row's top k rarely crowd more than 2 into
// one range (k = 32 over 57 ranges of 72 pages in the sparse workload), that
// key is T or close to it.  T0, its top 16 bits (half the
// search rounds), bounds T from below as well: only the keys >= T0 -- about k
// of them -- are searched.  The top-k grid starts behind the score grid with
// programmatic dependent launch, and releases its own successor at once (the
// next score grid's prefetch then overlaps this top-k).  They are compacted
// in page order; one warp ranks them against each other (up to 64, two per
// lane; beyond that it finds T two bits per round by warp reductions) and
// writes the chosen pages, ascending, with ties to the lower page index.  Many keys >= T0 (heavy
// ties) or rows longer than the registers hold take block-wide searches over
// every key.
#include <algorithm>

#include "common.cuh"

namespace argus {
namespace select {

constexpr int kScoreThreads = 256;
constexpr int kScoreCtasPerSm = 3;          // resident score CTAs per SM (register-limited)
constexpr int kTopkThreads = 512;
constexpr int kKeysPerThread = 8;             // top-k keys held in registers per thread
constexpr int kRowBatch = 8;               // compressed-key loads in flight per lane
constexpr int kTopkSmemKeys = 40 * 1024;   // rows up to this many pages are staged in shared memory
constexpr int kMaxPpc = 256;               // pages per score CTA (its keys per head in registers)
constexpr int kEmit = 2;                   // largest keys each score CTA reports per KV head
constexpr long long kScoreSmemBytes = 75 * 1024;   // a score CTA's shared memory (3 CTAs per SM)
constexpr int kPieceBytes = 16384;         // bulk-copy pieces of a score CTA's slab range, one mbarrier each
constexpr int kMaxPieces = 8;
static_assert(kScoreSmemBytes <= (long long)kPieceBytes * kMaxPieces, "one mbarrier per piece");

// Whether each score lane's rows all belong to one KV head (the rows per pass
// are a multiple of Hkv): its G-query sums then live in registers.
__host__ __device__ constexpr bool score_fixed_head(int D, int Hkv) {
  return ((kScoreThreads / 32) * (32 / (D / 8))) % Hkv == 0;
}

// Dynamic shared memory of a score CTA: its range's compressed keys, the
// G-query sums (only when lanes mix heads), the range's order keys, the
// pieces' mbarriers.
inline size_t score_smem_bytes(long long Hkv, long long D, long long ppc) {
  const size_t slab = ((size_t)ppc * Hkv * D * 2 + 127) / 128 * 128;
  const size_t qs = score_fixed_head((int)D, (int)Hkv) ? 0 : (size_t)Hkv * D * 4;
  return slab + qs + (size_t)((ppc * Hkv + 1) & ~1LL) * 4 + 8 * kMaxPieces;
}
constexpr int kSurvivorsPerLane = 16;      // keys >= T0 that one warp searches in registers

// Order-preserving map of an fp32 score to uint32: a > b  <=>  key(a) > key(b).
__device__ __forceinline__ uint32_t order_key(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// The kk-th largest of the values a warp holds (nv per lane; empty slots hold
// 0, which no candidate -- always >= 1 -- counts): two bits per round, the
// three candidate counts in two warp reductions.  No barrier.  (A key of 0 is
// the order key of a negative NaN score: NaN scores are unordered.)  With
// kLowBit > 0 the bits below kLowBit are left 0: the result is then the
// largest multiple of 2^kLowBit with at least kk values at or above it, a
// lower bound of the kk-th largest found in fewer rounds.
template <int NV, int kLowBit = 0>
__device__ __forceinline__ uint32_t warp_kth(const uint32_t (&vals)[NV], int kk) {
  uint32_t t = 0u;
  for (int bb = 30; bb >= kLowBit; bb -= 2) {
    const uint32_t c1 = t | (1u << bb), c2 = t | (2u << bb), c3 = t | (3u << bb);
    uint32_t a = 0u, c = 0u;
#pragma unroll
    for (int j = 0; j < NV; ++j) {
      a += (vals[j] >= c1 ? 1u : 0u) + (vals[j] >= c2 ? 0x10000u : 0u);
      c += vals[j] >= c3 ? 1u : 0u;
    }
    a = __reduce_add_sync(0xffffffffu, a);
    c = __reduce_add_sync(0xffffffffu, c);
    if (c >= (uint32_t)kk) t = c3;
    else if ((a >> 16) >= (uint32_t)kk) t = c2;
    else if ((a & 0xFFFFu) >= (uint32_t)kk) t = c1;
  }
  return t;
}

// The kEmit largest keys of each KV head over one score CTA's candidate pages
// (out of line: it runs once per CTA and keeps its registers apart from the
// scoring loop's).  Warp w takes KV heads w, w + 8, ...; lane l holds the keys
// of pages l + 32 m of the range (skeys [page][Hkv]); each round takes the
// warp's maximum and removes one instance of it.  out[h * stride + j], j <
// kEmit, gets the j-th largest key, or 0 past the range's n_loc candidates.
__device__ __noinline__ void local_top(const uint32_t* skeys, int Hkv, int n_loc, uint32_t* out, int stride) {
  const int lane = threadIdx.x & 31;
  for (int h = threadIdx.x >> 5; h < Hkv; h += kScoreThreads / 32) {
    uint32_t v[kMaxPpc / 32];
#pragma unroll
    for (int m = 0; m < kMaxPpc / 32; ++m) {
      const int lp = lane + 32 * m;
      v[m] = lp < n_loc ? skeys[lp * Hkv + h] : 0u;
    }
    for (int j = 0; j < kEmit; ++j) {
      uint32_t mx = 0u;
#pragma unroll
      for (int m = 0; m < kMaxPpc / 32; ++m) mx = max(mx, v[m]);
      const uint32_t top = __reduce_max_sync(0xffffffffu, mx);
      // the lowest lane holding it drops one instance
      const uint32_t holders = __ballot_sync(0xffffffffu, mx == top);
      if (top != 0u && lane == __ffs(holders) - 1) {
        bool done = false;
#pragma unroll
        for (int m = 0; m < kMaxPpc / 32; ++m) {
          if (!done && v[m] == top) {
            v[m] = 0u;
            done = true;
          }
        }
      }
      if (lane == 0) out[(size_t)h * stride + j] = top;
    }
  }
}

// Writes the order key of each page's score, [B][Hkv][max_pages] uint32, and
// (emit != NULL) each KV head's kEmit largest keys over the CTA's candidate
// pages (below n_cand(b) = n - 1 with keep_newest, else n),
// emit[B][Hkv][gridDim.x][kEmit], 0 where the range has fewer.
template <int D, bool QBF16>
__global__ void __launch_bounds__(kScoreThreads, kScoreCtasPerSm) score_kernel(int Hkv, int G, int max_pages, int ppc,
                                                              const void* __restrict__ q,
                                                              const uint16_t* __restrict__ ckeys,
                                                              const int32_t* __restrict__ n_pages,
                                                              uint32_t* __restrict__ keys, int keep_newest,
                                                              uint32_t* __restrict__ emit) {
  // the top-k grid may start its prologue now; it waits for this grid's keys
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // this grid itself may start during its stream predecessor's tail: every
  // input is read after that predecessor completes.  Before that, the CTA's
  // slab range and its batch row's queries are prefetched toward L2: a
  // prefetch only warms the cache (L2 is where the predecessor's writes land
  // too), so the bulk copies after the wait see the current bytes, sooner.
  if (threadIdx.x < 32) {
    const int pb = blockIdx.x * ppc, pe = min(max_pages, pb + ppc);
    const uint8_t* src = reinterpret_cast<const uint8_t*>(ckeys + (((size_t)blockIdx.y * max_pages + pb) * Hkv) * D);
    const uint32_t bytes = pb < pe ? (uint32_t)(pe - pb) * Hkv * D * 2 : 0u;
    for (uint32_t off = threadIdx.x * (uint32_t)kPieceBytes; off < bytes; off += 32u * kPieceBytes)
      asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src + off),
                   "r"(min((uint32_t)kPieceBytes, bytes - off))
                   : "memory");
    if (threadIdx.x == 0 && blockIdx.x == 0)
      asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(static_cast<const uint8_t*>(q) +
                                                                       (size_t)blockIdx.y * Hkv * G * D * 2),
                   "r"((uint32_t)(Hkv * G * D * 2))
                   : "memory");
  }
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // shared memory: the range's compressed keys [ppc * Hkv][D] bf16, the
  // G-query sums [Hkv][D] fp32, the range's order keys [ppc][Hkv], mbarriers
  extern __shared__ __align__(128) uint8_t sm_raw[];
  const size_t slab_bytes = ((size_t)ppc * Hkv * D * 2 + 127) / 128 * 128;
  const uint16_t* slab = reinterpret_cast<const uint16_t*>(sm_raw);
  const bool fixed_h = score_fixed_head(D, Hkv);
  float* qsum = reinterpret_cast<float*>(sm_raw + slab_bytes);   // [Hkv][D] when !fixed_h
  uint32_t* skeys = reinterpret_cast<uint32_t*>(qsum + (fixed_h ? 0 : Hkv * D));
  uint64_t* bars = reinterpret_cast<uint64_t*>(skeys + ((ppc * Hkv + 1) & ~1));
  const int b = blockIdx.y;
  const int p0 = blockIdx.x * ppc;
  const int Hq = Hkv * G;
  int n = n_pages[b];
  n = max(0, min(n, max_pages));
  const bool active = p0 < n;   // the range holds pages of the row
  constexpr int LPH = D / 8;               // lanes per (page, head) row, 16 bytes each
  constexpr int RPW = 32 / LPH;            // rows per warp and pass
  constexpr int RPP = (kScoreThreads / 32) * RPW;  // rows per CTA and pass
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int sub = lane / LPH, li = lane % LPH;
  const int p_end = active ? min(n, p0 + ppc) : p0;
  const int n_rows = (p_end - p0) * Hkv;
  const uint32_t total = (uint32_t)n_rows * D * 2;
  const int n_pieces = (int)((total + kPieceBytes - 1) / kPieceBytes);
  // rows of this CTA are contiguous in the slab: (p0 * Hkv + row) * D.  One
  // thread streams them into shared memory with bulk copies, 16 KB pieces on
  // an mbarrier each, while the other warps form the query sums: the whole
  // range is in flight at once, and scoring starts as soon as its first rows
  // have landed
  if (threadIdx.x == 0 && active) {
    for (int i = 0; i < n_pieces; ++i) mbar_init(&bars[i], 1);
    fence_mbar_init();
    const uint8_t* src = reinterpret_cast<const uint8_t*>(ckeys + (((size_t)b * max_pages + p0) * Hkv) * D);
    for (int i = 0; i < n_pieces; ++i) {
      const uint32_t off = (uint32_t)i * kPieceBytes, bytes = min((uint32_t)kPieceBytes, total - off);
      mbar_arrive_expect_tx(&bars[i], bytes);
      bulk_g2s(sm_raw + off, src + off, bytes, &bars[i]);
    }
  }
  uint4 x[kRowBatch];
  auto load_batch = [&](int r0) {
#pragma unroll
    for (int j = 0; j < kRowBatch; ++j) {
      const int row = r0 + j * RPP;
      if (row < n_rows) x[j] = *reinterpret_cast<const uint4*>(slab + (size_t)row * D + 8 * li);
      else x[j] = make_uint4(0u, 0u, 0u, 0u);
    }
  };
  const uint16_t* qb = static_cast<const uint16_t*>(q) + (size_t)b * Hq * D;
  // sum over the G query heads of head h of dims 8 c .. 8 c + 7; the rows'
  // 16-byte loads are issued together, eight at a time
  auto q_sum8 = [&](int h, int c, float (&acc)[8]) {
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = 0.f;
    for (int g0 = 0; g0 < G; g0 += 8) {
      uint4 xs[8];
#pragma unroll
      for (int u = 0; u < 8; ++u)
        xs[u] = (g0 + u < G) ? *reinterpret_cast<const uint4*>(qb + (size_t)(h * G + g0 + u) * D + 8 * c)
                             : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const uint32_t w[4] = {xs[u].x, xs[u].y, xs[u].z, xs[u].w};
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const uint32_t bits = (w[e / 2] >> (16 * (e & 1))) & 0xFFFFu;
          acc[e] += QBF16 ? __uint_as_float(bits << 16) : __half2float(__ushort_as_half((unsigned short)bits));
        }
      }
    }
  };
  // a lane whose rows share one KV head keeps that head's sums in registers;
  // otherwise the CTA forms every head's sums in shared memory
  float qv[8];
  if (fixed_h) {
    q_sum8((warp * RPW + sub) % Hkv, li, qv);
  } else {
    for (int idx = threadIdx.x; idx < Hkv * (D / 8); idx += blockDim.x) {
      const int h = idx / (D / 8), c = idx - h * (D / 8);
      float acc[8];
      q_sum8(h, c, acc);
#pragma unroll
      for (int e = 0; e < 8; ++e) qsum[h * D + 8 * c + e] = acc[e];
    }
  }
  __syncthreads();
  if (!active) return;   // no copy was issued
  static_assert(kRowBatch == 8, "the transposed reduction below folds 8 rows");
  int ready = 0;   // pieces known to have landed
  for (int r0 = warp * RPW + sub; r0 - sub < n_rows; r0 += kRowBatch * RPP) {
    // the pieces holding this warp's rows of the batch (a copy that never
    // completes leaves this CTA's keys unwritten rather than waiting forever)
    const int last_row = min(r0 - sub + (kRowBatch - 1) * RPP + RPW - 1, n_rows - 1);
    const int need = (int)(((uint32_t)(last_row + 1) * D * 2 - 1) / kPieceBytes);
    for (; ready <= need; ++ready)
      if (!mbar_wait(&bars[ready], 0)) return;
    load_batch(r0);
    float sv[kRowBatch];
#pragma unroll
    for (int j = 0; j < kRowBatch; ++j) {
      const int row = r0 + j * RPP;
      float qe[8];
      if (fixed_h) {
#pragma unroll
        for (int e = 0; e < 8; ++e) qe[e] = qv[e];
      } else {
        const float* qs = qsum + (row % Hkv) * D + 8 * li;
#pragma unroll
        for (int e = 0; e < 8; ++e) qe[e] = qs[e];
      }
      const uint32_t w[4] = {x[j].x, x[j].y, x[j].z, x[j].w};
      float acc = 0.f;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float k = __uint_as_float(((w[e / 2] >> (16 * (e & 1))) & 0xFFFFu) << 16);
        acc = fmaf(k, qe[e], acc);
      }
      sv[j] = acc;
    }
    // transposed reduction over the row's LPH lanes: each step halves the
    // values a lane holds (8 -> 4 -> 2 -> 1), then plain sums finish
    float v4[4], v2[2], v1;
    {
      constexpr int o = LPH / 2;
      const bool up = (li & o) != 0;
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        const float mine = up ? sv[v + 4] : sv[v], other = up ? sv[v] : sv[v + 4];
        v4[v] = mine + __shfl_xor_sync(0xffffffffu, other, o);
      }
    }
    {
      constexpr int o = LPH / 4;
      const bool up = (li & o) != 0;
#pragma unroll
      for (int v = 0; v < 2; ++v) {
        const float mine = up ? v4[v + 2] : v4[v], other = up ? v4[v] : v4[v + 2];
        v2[v] = mine + __shfl_xor_sync(0xffffffffu, other, o);
      }
    }
    {
      constexpr int o = LPH / 8;
      const bool up = (li & o) != 0;
      const float mine = up ? v2[1] : v2[0], other = up ? v2[0] : v2[1];
      v1 = mine + __shfl_xor_sync(0xffffffffu, other, o);
    }
#pragma unroll
    for (int o = LPH / 16; o >= 1; o >>= 1) v1 += __shfl_xor_sync(0xffffffffu, v1, o);
    // this lane now holds the sum of row j, the bits of j chosen by the steps above
    const int j = ((li & (LPH / 2)) ? 4 : 0) + ((li & (LPH / 4)) ? 2 : 0) + ((li & (LPH / 8)) ? 1 : 0);
    const int row = r0 + j * RPP;
    // (with LPH = 16, lanes li and li ^ 1 hold the same row: the even one writes)
    if ((LPH == 8 || (li & 1) == 0) && row < n_rows) {
      const int p = p0 + row / Hkv;
      const uint32_t key = order_key(v1);
      keys[((size_t)b * Hkv + row % Hkv) * max_pages + p] = key;
      skeys[row] = key;
    }
  }
  if (emit == nullptr) return;
  __syncthreads();
  const int n_cand = keep_newest ? n - 1 : n;
  local_top(skeys, Hkv, max(0, min(p_end, n_cand) - p0),
            emit + ((size_t)b * Hkv * gridDim.x + blockIdx.x) * kEmit, gridDim.x * kEmit);
}

// Exclusive block-wide prefix sum of one int per thread; returns the total.
__device__ __forceinline__ int block_exclusive_scan(int v, int* sh, int& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  __syncthreads();
  if (lane == 31) sh[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = (lane < (int)(blockDim.x >> 5)) ? sh[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    sh[lane] = w;  // inclusive warp totals
  }
  __syncthreads();
  total = sh[(blockDim.x >> 5) - 1];
  const int before = (warp > 0) ? sh[warp - 1] : 0;
  return before + x - v;
}

// One CTA per (KV head, batch row).  The row's keys are staged in shared
// memory when stage != 0 (dynamic shared memory of max_pages words).  emit:
// the score kernel's largest keys per page range (n_chunks ranges of ppc
// pages per row, kEmit keys each).
__global__ void __launch_bounds__(kTopkThreads) topk_kernel(int Hkv, int max_pages, const uint32_t* keys_g,
                                                            const int32_t* n_pages, int top_k, int keep_newest,
                                                            int32_t* sel_pages, int32_t* sel_count, int width,
                                                            uint32_t* drops, int stage, const uint32_t* emit_g,
                                                            int n_chunks, int ppc) {
  extern __shared__ uint32_t skeys[];
  __shared__ int sh_scan[32];
  __shared__ uint2 sh_cnt2[2][32];
  __shared__ uint32_t sh_t0;
  __shared__ uint32_t sh_cand[kKeysPerThread * kTopkThreads];   // keys >= T0, in page order
  __shared__ uint16_t sh_page[kKeysPerThread * kTopkThreads];   // their pages
  const int h = blockIdx.x, b = blockIdx.y;
  const int tid = threadIdx.x, nthr = blockDim.x;
  const int lane = tid & 31, warp = tid >> 5;
  int n = n_pages[b];
  const int n_raw = n;
  n = max(0, min(n, max_pages));
  int32_t* out = sel_pages + ((size_t)b * Hkv + h) * width;
  const uint32_t* keys = keys_g + ((size_t)b * Hkv + h) * max_pages;
  uint32_t dropped = 0;
  if (n_raw > max_pages && tid == 0 && h == 0) dropped += (uint32_t)(n_raw - max_pages);
  const int n_cand = (n > 0) ? (keep_newest ? n - 1 : n) : 0;
  const int room = width - ((keep_newest && n > 0) ? 1 : 0);
  const int k_want = min(top_k, n_cand);
  const int k = max(0, min(k_want, room));
  if (tid == 0) dropped += (uint32_t)(k_want - k);
  // launched behind the score grid with programmatic dependent launch: its
  // keys are read after this wait.  Its own successor may start now (a decode
  // or the next score grid waits for this grid before reading its results).
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  constexpr int KPT = kKeysPerThread;
  const bool in_regs = n_cand <= KPT * nthr;
  const bool search = k > 0 && k < n_cand;

  // ---- fast path: the keys >= T0, in page order, searched by one warp
  if (search && in_regs) {
    // thread t holds pages [KPT t, KPT t + KPT): page order is (thread, slot)
    uint32_t kr[KPT];
#pragma unroll
    for (int j = 0; j < KPT; ++j) {
      const int pk = KPT * tid + j;
      kr[j] = pk < n_cand ? keys[pk] : 0u;
    }
    // T0 <= the k-th largest of the keys the ranges reported (real keys of
    // distinct pages), so T0 <= T, the row's k-th largest: its top 16 bits,
    // which also admits the few keys just below it in the same 16-bit bucket
    // (0 when the report is too long to hold, or holds fewer than k keys)
    // (warp 0 alone, then one barrier)
    const int n_ranges = min(n_chunks, (n_cand + ppc - 1) / ppc);
    const int n_emit = n_ranges * kEmit;
    if (warp == 0) {
      uint32_t t0w = 0u;
      const uint32_t* er = emit_g + ((size_t)b * Hkv + h) * n_chunks * kEmit;
      if (n_emit >= k && n_emit <= 128) {   // four per lane
        uint32_t ev[4];
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          const int i = lane + 32 * m;
          ev[m] = i < n_emit ? er[i] : 0u;
        }
        t0w = warp_kth<4, 16>(ev, k);
      } else if (n_emit >= k && n_emit <= 256) {   // eight per lane
        uint32_t ev[8];
#pragma unroll
        for (int m = 0; m < 8; ++m) {
          const int i = lane + 32 * m;
          ev[m] = i < n_emit ? er[i] : 0u;
        }
        t0w = warp_kth<8, 16>(ev, k);
      } else if (n_emit >= k && n_emit <= 32 * kSurvivorsPerLane) {
        uint32_t ev[kSurvivorsPerLane];
#pragma unroll
        for (int m = 0; m < kSurvivorsPerLane; ++m) {
          const int i = lane + 32 * m;
          ev[m] = i < n_emit ? er[i] : 0u;
        }
        t0w = warp_kth<kSurvivorsPerLane, 16>(ev, k);
      }
      if (lane == 0) sh_t0 = t0w;
    }
    __syncthreads();
    const uint32_t t0 = sh_t0;
    int my = 0;
#pragma unroll
    for (int j = 0; j < KPT; ++j) my += (KPT * tid + j < n_cand && kr[j] >= t0) ? 1 : 0;
    int M;
    int pos = block_exclusive_scan(my, sh_scan, M);
    if (M <= 32 * kSurvivorsPerLane) {
#pragma unroll
      for (int j = 0; j < KPT; ++j) {
        const int pk = KPT * tid + j;
        if (pk < n_cand && kr[j] >= t0) {
          sh_cand[pos] = kr[j];
          sh_page[pos] = (uint16_t)pk;
          ++pos;
        }
      }
      __syncthreads();
      if (warp == 0) {
        // survivor i = lane + 32 m: index order is page order
        const uint32_t below = (1u << lane) - 1u;
        int written = 0;
        if (M <= 64) {
          // the usual case, about k survivors, two per lane: each is ranked
          // against all the others, rank_i = #{j : c_j > c_i} + #{j < i :
          // c_j == c_i} (a permutation of 0 .. M-1); the k survivors of rank
          // below k are the row's top k, ties to the lower page
          const uint32_t x0 = lane < M ? sh_cand[lane] : 0u;
          const uint32_t x1 = lane + 32 < M ? sh_cand[lane + 32] : 0u;
          int r0 = 0, r1 = 0;
#pragma unroll 8
          for (int src = 0; src < 32; ++src) {
            const uint32_t y0 = __shfl_sync(0xffffffffu, x0, src);   // survivor src
            const uint32_t y1 = __shfl_sync(0xffffffffu, x1, src);   // survivor src + 32
            const bool v0 = src < M, v1 = src + 32 < M;
            r0 += ((v0 && (y0 > x0 || (y0 == x0 && src < lane))) ? 1 : 0) + ((v1 && y1 > x0) ? 1 : 0);
            r1 += ((v0 && y0 >= x1) ? 1 : 0) + ((v1 && (y1 > x1 || (y1 == x1 && src < lane))) ? 1 : 0);
          }
          const bool take0 = lane < M && r0 < k, take1 = lane + 32 < M && r1 < k;
          const uint32_t b0 = __ballot_sync(0xffffffffu, take0), b1 = __ballot_sync(0xffffffffu, take1);
          if (take0) out[__popc(b0 & below)] = sh_page[lane];
          if (take1) out[__popc(b0) + __popc(b1 & below)] = sh_page[lane + 32];
          written = __popc(b0) + __popc(b1);
        } else {
          uint32_t cv[kSurvivorsPerLane];
#pragma unroll
          for (int m = 0; m < kSurvivorsPerLane; ++m) {
            const int i = lane + 32 * m;
            cv[m] = i < M ? sh_cand[i] : 0u;
          }
          const uint32_t T = warp_kth(cv, k);
          uint32_t gt = 0u;
#pragma unroll
          for (int m = 0; m < kSurvivorsPerLane; ++m) gt += cv[m] > T ? 1u : 0u;
          gt = __reduce_add_sync(0xffffffffu, gt);
          const int k_rem = k - (int)gt;   // ties at T taken, lowest pages first
          int ties_seen = 0;
#pragma unroll
          for (int m = 0; m < kSurvivorsPerLane; ++m) {
            const int i = lane + 32 * m;
            const bool tie = i < M && cv[m] == T;
            const uint32_t tb = __ballot_sync(0xffffffffu, tie);
            const bool take = (i < M && cv[m] > T) || (tie && ties_seen + __popc(tb & below) < k_rem);
            const uint32_t kb = __ballot_sync(0xffffffffu, take);
            if (take) out[written + __popc(kb & below)] = sh_page[i];
            written += __popc(kb);
            ties_seen += __popc(tb);
          }
        }
        // written == k <= room; the newest page (larger than every candidate) last
        int total = written;
        if (keep_newest && n > 0) {
          if (lane == 0) out[total] = n - 1;
          ++total;
        }
        for (int i = total + lane; i < width; i += 32) out[i] = -1;
        if (lane == 0) {
          sel_count[(size_t)b * Hkv + h] = total;
          if (dropped && drops) atomicAdd(drops, dropped);
        }
      }
      return;
    }
    __syncthreads();   // many ties: fall through to the block-wide search
  }

  if (stage) {  // eight loads in flight per thread
    for (int p0 = 0; p0 < n_cand; p0 += 8 * nthr) {
      uint32_t v[8];
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const int pk = p0 + kk * nthr + tid;
        v[kk] = pk < n_cand ? keys[pk] : 0u;
      }
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const int pk = p0 + kk * nthr + tid;
        if (pk < n_cand) skeys[pk] = v[kk];
      }
    }
    keys = skeys;
    __syncthreads();
  }

  // Block-wide threshold: T = the k-th largest key, found bit by bit from the
  // top as the largest value with at least k keys >= T (block-wide counts:
  // per-warp reductions, double-buffered partial sums, one barrier per two
  // bits).  All keys > T are taken, and the first k_rem (in page order) equal to T.
  uint32_t T = 0u;
  int k_rem = 0;
  if (search) {
    uint32_t kr[KPT];
    bool kv[KPT];
#pragma unroll
    for (int j = 0; j < KPT; ++j) {
      const int pk = tid + j * nthr;
      kv[j] = in_regs && pk < n_cand;
      kr[j] = kv[j] ? keys[pk] : 0u;
    }
    // counts of keys >= a, >= b (strict: > a) packed as two 16-bit fields
    // (a row has at most 65535 candidates), one reduction
    auto count2 = [&](uint32_t a, uint32_t bnd, bool strict) -> uint32_t {
      uint32_t c = 0;
      if (in_regs) {
#pragma unroll
        for (int j = 0; j < KPT; ++j)
          c += kv[j] ? ((strict ? kr[j] > a : kr[j] >= a) ? 1u : 0u) + (kr[j] >= bnd ? 0x10000u : 0u) : 0u;
      } else {
        for (int pk = tid; pk < n_cand; pk += nthr) {
          const uint32_t x = keys[pk];
          c += ((strict ? x > a : x >= a) ? 1u : 0u) + (x >= bnd ? 0x10000u : 0u);
        }
      }
      return __reduce_add_sync(0xffffffffu, c);
    };
    // block totals of two packed words: each warp posts its pair, then every
    // warp sums the posts (one per lane) -- one barrier per round, the two
    // buffers alternate
    auto block_total2 = [&](uint32_t c0, uint32_t c1, int buf) -> uint2 {
      if (lane == 0) sh_cnt2[buf][warp] = make_uint2(c0, c1);
      __syncthreads();
      const uint2 x = lane < (nthr >> 5) ? sh_cnt2[buf][lane] : make_uint2(0u, 0u);
      return make_uint2(__reduce_add_sync(0xffffffffu, x.x), __reduce_add_sync(0xffffffffu, x.y));
    };
    for (int bb = 30, round = 0; bb >= 0; bb -= 2, ++round) {
      const uint32_t c1 = T | (1u << bb), c2 = T | (2u << bb), c3 = T | (3u << bb);
      const uint2 cnt = block_total2(count2(c1, c2, false), count2(c3, 0xFFFFFFFFu, false), round & 1);
      if ((cnt.y & 0xFFFFu) >= (uint32_t)k) T = c3;
      else if ((cnt.x >> 16) >= (uint32_t)k) T = c2;
      else if ((cnt.x & 0xFFFFu) >= (uint32_t)k) T = c1;
    }
    // the last round (15) used buffer 1, so 0 is free
    k_rem = k - (int)(block_total2(count2(T, 0xFFFFFFFFu, true), 0u, 0).x & 0xFFFFu);
  }
  const bool take_all = (k >= n_cand);
  // per thread: a contiguous range of pages so that scans keep page order
  const int per = (n + nthr - 1) / nthr;
  const int lo = min(n, tid * per), hi = min(n, lo + per);
  int ties = 0;
  if (!take_all && k > 0) {
    for (int p = lo; p < min(hi, n_cand); ++p) ties += (keys[p] == T);
  }
  int tie_total;
  const int tie_start = block_exclusive_scan(ties, sh_scan, tie_total);
  auto take_of = [&](int p, int& tie_before) -> bool {
    if (p >= n_cand) return keep_newest && p == n - 1;
    if (take_all) return true;
    if (k == 0) return false;
    const uint32_t key = keys[p];
    if (key > T) return true;
    if (key == T) return tie_before++ < k_rem;
    return false;
  };
  int mine = 0, tb = tie_start;
  for (int p = lo; p < hi; ++p) mine += take_of(p, tb);
  int total;
  int pos = block_exclusive_scan(mine, sh_scan, total);
  tb = tie_start;
  for (int p = lo; p < hi; ++p) {
    if (take_of(p, tb) && pos < width) out[pos++] = p;
  }
  for (int i = total + tid; i < width; i += nthr) out[i] = -1;
  if (tid == 0) {
    sel_count[(size_t)b * Hkv + h] = min(total, width);
    if (dropped && drops) atomicAdd(drops, dropped);
  }
}

}  // namespace select
}  // namespace argus

using namespace argus;

// Workspace: the order keys [B][Hkv][max_pages], then the reported largest
// keys [B][Hkv][chunks][kEmit] for at most ceil(max_pages / 8) page ranges
// (ranges hold at least 8 pages), so that the size does not depend on the
// device.
static size_t select_ws(long long batch, long long n_kv_heads, long long max_pages) {
  const size_t keys = (size_t)batch * n_kv_heads * max_pages * sizeof(uint32_t);
  return keys + (size_t)batch * n_kv_heads * ((max_pages + 7) / 8) * select::kEmit * sizeof(uint32_t);
}

extern "C" argus_status argus_select_workspace_bytes(const argus_geom* g, int32_t batch, int32_t max_pages,
                                                     size_t* bytes) {
  if (!g || !bytes) return fail(ARGUS_E_INVALID, "select: NULL argument");
  if (batch < 0 || max_pages < 0 || g->n_kv_heads <= 0) return fail(ARGUS_E_INVALID, "select: bad sizes");
  *bytes = select_ws(batch, g->n_kv_heads, max_pages);
  return ARGUS_OK;
}

extern "C" argus_status argus_select_pages(const argus_geom* g, int32_t batch, const void* q, int32_t q_dtype,
                                           const void* ckeys, const int32_t* n_pages, int32_t max_pages,
                                           int32_t top_k, int32_t keep_newest, int32_t* sel_pages,
                                           int32_t* sel_count, int32_t sel_width, uint32_t* drop_counter,
                                           void* ws, size_t ws_bytes, void* stream) {
  if (!g) return fail(ARGUS_E_INVALID, "select: geometry is NULL");
  if (g->n_q_heads <= 0 || g->n_kv_heads <= 0 || g->n_q_heads % g->n_kv_heads)
    return fail(ARGUS_E_INVALID, "select: bad head counts");
  if (g->head_dim != 64 && g->head_dim != 128)
    return fail(ARGUS_E_UNSUPPORTED, "select: head_dim %d (supported: 64, 128)", g->head_dim);
  if (q_dtype != ARGUS_FP16 && q_dtype != ARGUS_BF16) return fail(ARGUS_E_INVALID, "select: q_dtype");
  if (batch < 0 || max_pages <= 0 || top_k < 0 || sel_width <= 0)
    return fail(ARGUS_E_INVALID, "select: bad batch / max_pages / top_k / sel_width");
  if (batch > 65535 || g->n_kv_heads > 65535) return fail(ARGUS_E_UNSUPPORTED, "select: grid too large");
  if (max_pages > 65535) return fail(ARGUS_E_UNSUPPORTED, "select: max_pages %d (at most 65535)", max_pages);
  if (batch == 0) return ARGUS_OK;
  if (!q || !ckeys || !n_pages || !sel_pages || !sel_count)
    return fail(ARGUS_E_INVALID, "select: NULL pointer");
  if ((reinterpret_cast<uintptr_t>(ckeys) | reinterpret_cast<uintptr_t>(q)) & 15)
    return fail(ARGUS_E_INVALID, "select: q and ckeys must be 16-byte aligned");
  size_t need = select_ws(batch, g->n_kv_heads, max_pages);
  if (!ws || ws_bytes < need) return fail(ARGUS_E_WORKSPACE, "select: workspace %zu < %zu", ws_bytes, need);
  if (reinterpret_cast<uintptr_t>(ws) & 3) return fail(ARGUS_E_INVALID, "select: workspace not 4-byte aligned");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int G = g->n_q_heads / g->n_kv_heads;
  uint32_t* keys = static_cast<uint32_t*>(ws);
  uint32_t* emit = keys + (size_t)batch * g->n_kv_heads * max_pages;
  // pages per CTA: the whole slab in one wave of resident CTAs, 8 .. 256 pages,
  // as long as a CTA's shared memory stays within kScoreSmemBytes (three per SM)
  const long long resident = (long long)device_sm_count() * select::kScoreCtasPerSm;
  long long ppc = ((long long)batch * max_pages + resident - 1) / resident;
  ppc = std::min<long long>(select::kMaxPpc, std::max<long long>(8, (ppc + 7) / 8 * 8));
  while (ppc > 8 && (long long)select::score_smem_bytes(g->n_kv_heads, g->head_dim, ppc) > select::kScoreSmemBytes)
    ppc -= 8;
  const int n_chunks = (int)((max_pages + ppc - 1) / ppc);
  dim3 grid1((unsigned)n_chunks, batch);
  const size_t sh = select::score_smem_bytes(g->n_kv_heads, g->head_dim, ppc);
  if (sh > 227 * 1024) return fail(ARGUS_E_UNSUPPORTED, "select: n_kv_heads * head_dim too large");
  {
    static PerContext configured;
    argus_status sta = configured.ensure([](int) {
      cudaError_t e = cudaSuccess;
      const int mx = 227 * 1024;
      if (e == cudaSuccess) e = cudaFuncSetAttribute(select::score_kernel<64, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, mx);
      if (e == cudaSuccess) e = cudaFuncSetAttribute(select::score_kernel<64, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, mx);
      if (e == cudaSuccess) e = cudaFuncSetAttribute(select::score_kernel<128, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, mx);
      if (e == cudaSuccess) e = cudaFuncSetAttribute(select::score_kernel<128, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, mx);
      if (e != cudaSuccess) return fail(ARGUS_E_LAUNCH, "select: score smem attribute: %s", cudaGetErrorString(e));
      return ARGUS_OK;
    });
    if (sta != ARGUS_OK) return sta;
  }
  uint32_t* emit_arg = top_k > 0 ? emit : nullptr;
  const uint16_t* ck = static_cast<const uint16_t*>(ckeys);
  const bool bf = (q_dtype == ARGUS_BF16);
  const int kn = keep_newest ? 1 : 0;
  {
    // programmatic dependent launch: the score grid starts during its stream
    // predecessor's tail and waits for it before reading anything
    cudaLaunchConfig_t sc = {};
    sc.gridDim = grid1;
    sc.blockDim = dim3(select::kScoreThreads);
    sc.dynamicSmemBytes = sh;
    sc.stream = s;
    cudaLaunchAttribute sattr[1];
    sattr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    sattr[0].val.programmaticStreamSerializationAllowed = 1;
    sc.attrs = sattr;
    sc.numAttrs = 1;
    const int Hkv_i = g->n_kv_heads, mp = max_pages, ppc_i = (int)ppc;
    cudaError_t se;
    if (g->head_dim == 64) {
      se = bf ? cudaLaunchKernelEx(&sc, select::score_kernel<64, true>, Hkv_i, G, mp, ppc_i, q, ck, n_pages, keys, kn, emit_arg)
              : cudaLaunchKernelEx(&sc, select::score_kernel<64, false>, Hkv_i, G, mp, ppc_i, q, ck, n_pages, keys, kn, emit_arg);
    } else {
      se = bf ? cudaLaunchKernelEx(&sc, select::score_kernel<128, true>, Hkv_i, G, mp, ppc_i, q, ck, n_pages, keys, kn, emit_arg)
              : cudaLaunchKernelEx(&sc, select::score_kernel<128, false>, Hkv_i, G, mp, ppc_i, q, ck, n_pages, keys, kn, emit_arg);
    }
    if (se != cudaSuccess) return fail(ARGUS_E_LAUNCH, "argus_select_pages (score): %s", cudaGetErrorString(se));
  }
  argus_status st = launch_status("argus_select_pages (score)");
  if (st != ARGUS_OK) return st;
  const int stage = max_pages <= select::kTopkSmemKeys ? 1 : 0;
  const size_t tsh = stage ? (size_t)max_pages * sizeof(uint32_t) : 0;
  if (tsh > 48 * 1024) {
    static PerContext configured;
    argus_status sta = configured.ensure([](int) {
      cudaError_t e = cudaFuncSetAttribute(select::topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           select::kTopkSmemKeys * (int)sizeof(uint32_t));
      if (e != cudaSuccess) return fail(ARGUS_E_LAUNCH, "select: smem attribute: %s", cudaGetErrorString(e));
      return ARGUS_OK;
    });
    if (sta != ARGUS_OK) return sta;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(g->n_kv_heads, batch);
  cfg.blockDim = dim3(select::kTopkThreads);
  cfg.dynamicSmemBytes = tsh;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, select::topk_kernel, g->n_kv_heads, max_pages, (const uint32_t*)keys,
                                     n_pages, top_k, (int)keep_newest, sel_pages, sel_count, sel_width, drop_counter,
                                     stage, (const uint32_t*)emit, n_chunks, (int)ppc);
  if (e != cudaSuccess) return fail(ARGUS_E_LAUNCH, "argus_select_pages (top-k): %s", cudaGetErrorString(e));
  return launch_status("argus_select_pages (top-k)");
}
