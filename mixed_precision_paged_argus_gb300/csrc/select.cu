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
// (D bf16 per page and head); one wave of CTAs tiles (batch row, page range),
// lanes read 16 bytes of a compressed key each, eight rows' loads in flight,
// and fold eight rows' partial dot products across the head's lanes in one
// transposed reduction; the G-query sum is formed once per CTA and kept in
// registers; scores are stored as order-preserving uint32 keys.
// (2) top-k: one CTA per (batch row, KV head) stages the row's keys in shared
// memory and registers; each warp narrows its keys to those at or above its
// own k-th largest, the k-th largest of the survivors is the row's threshold
// (both searches two bits per round by warp reductions), then the chosen
// pages are compacted in ascending order with block-wide prefix sums.
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

// Order-preserving map of an fp32 score to uint32: a > b  <=>  key(a) > key(b).
__device__ __forceinline__ uint32_t order_key(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Writes the order key of each page's score, [B][Hkv][max_pages] uint32.
template <int D, bool QBF16>
__global__ void __launch_bounds__(kScoreThreads) score_kernel(int Hkv, int G, int max_pages, int ppc,
                                                              const void* __restrict__ q,
                                                              const uint16_t* __restrict__ ckeys,
                                                              const int32_t* __restrict__ n_pages,
                                                              uint32_t* __restrict__ keys) {
  extern __shared__ float qsum[];  // [Hkv][D]
  const int b = blockIdx.y;
  const int p0 = blockIdx.x * ppc;
  const int Hq = Hkv * G;
  int n = n_pages[b];
  n = max(0, min(n, max_pages));
  if (p0 >= n) return;
  constexpr int LPH = D / 8;               // lanes per (page, head) row, 16 bytes each
  constexpr int RPW = 32 / LPH;            // rows per warp and pass
  constexpr int RPP = (kScoreThreads / 32) * RPW;  // rows per CTA and pass
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int sub = lane / LPH, li = lane % LPH;
  const int p_end = min(n, p0 + ppc);
  const int n_rows = (p_end - p0) * Hkv;
  // rows of this CTA are contiguous in the slab: (p0 * Hkv + row) * D
  const uint16_t* base = ckeys + (((size_t)b * max_pages + p0) * Hkv) * D + 8 * li;
  // the first batch of rows does not depend on the q sums: its loads go out
  // before them, so the two latencies overlap
  uint4 x[kRowBatch];
  auto load_batch = [&](int r0) {
#pragma unroll
    for (int j = 0; j < kRowBatch; ++j) {
      const int row = r0 + j * RPP;
      if (row < n_rows) x[j] = __ldcs(reinterpret_cast<const uint4*>(base + (size_t)row * D));
      else x[j] = make_uint4(0u, 0u, 0u, 0u);
    }
  };
  load_batch(warp * RPW + sub);
  const uint16_t* qb = static_cast<const uint16_t*>(q) + (size_t)b * Hq * D;
  // G-query sums: a thread per (KV head, 8 dims); the rows' 16-byte loads are
  // issued together, eight at a time
  for (int idx = threadIdx.x; idx < Hkv * (D / 8); idx += blockDim.x) {
    const int h = idx / (D / 8), c = idx - h * (D / 8);
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
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
#pragma unroll
    for (int e = 0; e < 8; ++e) qsum[h * D + 8 * c + e] = acc[e];
  }
  __syncthreads();
  // when Hkv divides the rows per pass, a lane's rows all belong to one KV
  // head: its 8 q-sum values stay in registers
  const bool fixed_h = (RPP % Hkv) == 0;
  float qv[8];
  {
    const int h0 = (warp * RPW + sub) % Hkv;
#pragma unroll
    for (int e = 0; e < 8; ++e) qv[e] = qsum[h0 * D + 8 * li + e];
  }
  static_assert(kRowBatch == 8, "the transposed reduction below folds 8 rows");
  for (int r0 = warp * RPW + sub; r0 - sub < n_rows; r0 += kRowBatch * RPP) {
    if (r0 != warp * RPW + sub) load_batch(r0);   // the first batch is already loaded
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
      keys[((size_t)b * Hkv + row % Hkv) * max_pages + p] = order_key(v1);
    }
  }
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
// memory when stage != 0 (dynamic shared memory of max_pages words).
__global__ void __launch_bounds__(kTopkThreads) topk_kernel(int Hkv, int max_pages, const uint32_t* keys_g,
                                                            const int32_t* n_pages, int top_k, int keep_newest,
                                                            int32_t* sel_pages, int32_t* sel_count, int width,
                                                            uint32_t* drops, int stage) {
  extern __shared__ uint32_t skeys[];
  __shared__ int sh_scan[32];
  __shared__ uint2 sh_cnt2[2][32];
  __shared__ int sh_wc[32];
  __shared__ uint32_t sh_thr[2];
  __shared__ uint32_t sh_cand[kKeysPerThread * kTopkThreads];   // survivors of the per-warp search
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
  if (stage) {  // eight loads in flight per thread
    for (int p0 = 0; p0 < n_cand; p0 += 8 * nthr) {
      uint32_t v[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int pk = p0 + k * nthr + tid;
        v[k] = pk < n_cand ? keys[pk] : 0u;
      }
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int pk = p0 + k * nthr + tid;
        if (pk < n_cand) skeys[pk] = v[k];
      }
    }
    keys = skeys;
    __syncthreads();
  }

  // Threshold: T = the k-th largest key, found bit by bit from the top as the
  // largest value with at least k keys >= T (block-wide counts: per-warp
  // reductions, double-buffered partial sums, one barrier per bit).  All keys
  // > T are taken, and the first k_rem (in page order) equal to T.
  const uint32_t mask = 0xFFFFFFFFu;
  uint32_t T = 0u;
  int k_rem = 0;
  if (k > 0 && k < n_cand) {
    // up to kKeysPerThread keys per thread live in registers; longer rows are
    // re-read from memory every bit
    constexpr int KPT = kKeysPerThread;
    const bool in_regs = n_cand <= KPT * nthr;
    uint32_t kr[KPT];
    bool kv[KPT];
#pragma unroll
    for (int j = 0; j < KPT; ++j) {
      const int pk = tid + j * nthr;
      kv[j] = in_regs && pk < n_cand;
      kr[j] = kv[j] ? keys[pk] : 0u;
    }
    // counts of keys >= a, >= b (strict: > a) packed as two 16-bit fields
    // (a row has at most kTopkSmemKeys < 2^16 candidates), one reduction
    auto count2 = [&](uint32_t a, uint32_t b, bool strict) -> uint32_t {
      uint32_t c = 0;
      if (in_regs) {
#pragma unroll
        for (int j = 0; j < KPT; ++j)
          c += kv[j] ? ((strict ? kr[j] > a : kr[j] >= a) ? 1u : 0u) + (kr[j] >= b ? 0x10000u : 0u) : 0u;
      } else {
        for (int pk = tid; pk < n_cand; pk += nthr) {
          const uint32_t x = keys[pk];
          c += ((strict ? x > a : x >= a) ? 1u : 0u) + (x >= b ? 0x10000u : 0u);
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
    // Warp-level search for the kk-th largest of the values a warp holds
    // (nv per lane in registers, valid flags vf): two bits per round, the
    // three candidate counts in two warp reductions.  No barrier.
    // Empty slots hold 0, which no candidate (always >= 1) counts.  (A key of 0
    // is the order key of a negative NaN score: NaN scores are unordered.)
    auto warp_kth = [&](const uint32_t* vals, int nv, int kk) -> uint32_t {
      uint32_t t = 0u;
      for (int bb = 30; bb >= 0; bb -= 2) {
        const uint32_t c1 = t | (1u << bb), c2 = t | (2u << bb), c3 = t | (3u << bb);
        uint32_t a = 0u, c = 0u;
        for (int j = 0; j < nv; ++j) {
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
    };
    if (in_regs) {
      // (1) each warp keeps its keys >= its own min(k, n_w)-th largest: every
      // key >= the row's k-th largest survives, so (2) the row's threshold is
      // the k-th largest of the survivors, found by every warp alike
      int nw_valid = 0;
#pragma unroll
      for (int j = 0; j < KPT; ++j) nw_valid += kv[j] ? 1 : 0;
      nw_valid = (int)__reduce_add_sync(0xffffffffu, (uint32_t)nw_valid);
      const int kw = min(k, nw_valid);
      const uint32_t Tw = kw > 0 ? warp_kth(kr, KPT, kw) : 0xFFFFFFFFu;
      int my = 0;
#pragma unroll
      for (int j = 0; j < KPT; ++j) my += (kv[j] && kw > 0 && kr[j] >= Tw) ? 1 : 0;
      int incl = my;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      if (lane == 31) sh_wc[warp] = incl;
      __syncthreads();
      const int nwarps = nthr >> 5;
      const int wcl = lane < nwarps ? sh_wc[lane] : 0;
      const int M = (int)__reduce_add_sync(0xffffffffu, (uint32_t)wcl);
      const int wbase = (int)__reduce_add_sync(0xffffffffu, (uint32_t)(lane < warp ? wcl : 0));
      int pos = wbase + incl - my;
#pragma unroll
      for (int j = 0; j < KPT; ++j)
        if (kv[j] && kw > 0 && kr[j] >= Tw) sh_cand[pos++] = kr[j];
      __syncthreads();
      constexpr int CPL = 16;   // survivors per lane held in registers
      if (M <= 32 * CPL) {
        // one warp searches the survivors; the others wait for its answer
        if (warp == 0) {
          uint32_t cv[CPL];
#pragma unroll
          for (int m = 0; m < CPL; ++m) {
            const int i = lane + 32 * m;
            cv[m] = i < M ? sh_cand[i] : 0u;
          }
          const uint32_t t = warp_kth(cv, CPL, k);
          uint32_t gt = 0u;
#pragma unroll
          for (int m = 0; m < CPL; ++m) gt += cv[m] > t ? 1u : 0u;
          gt = __reduce_add_sync(0xffffffffu, gt);
          if (lane == 0) {
            sh_thr[0] = t;
            sh_thr[1] = (uint32_t)(k - (int)gt);
          }
        }
        __syncthreads();
        T = sh_thr[0];
        k_rem = (int)sh_thr[1];
      } else {
        // many survivors (ties): block-wide search over every key
        for (int b = 30, round = 0; b >= 0; b -= 2, ++round) {
          const uint32_t c1 = T | (1u << b), c2 = T | (2u << b), c3 = T | (3u << b);
          const uint2 n = block_total2(count2(c1, c2, false), count2(c3, 0xFFFFFFFFu, false), round & 1);
          if ((n.y & 0xFFFFu) >= (uint32_t)k) T = c3;
          else if ((n.x >> 16) >= (uint32_t)k) T = c2;
          else if ((n.x & 0xFFFFu) >= (uint32_t)k) T = c1;
        }
        k_rem = k - (int)(block_total2(count2(T, 0xFFFFFFFFu, true), 0u, 0).x & 0xFFFFu);
      }
    } else {
      // rows longer than the registers hold: block-wide search, two bits per round
      for (int b = 30, round = 0; b >= 0; b -= 2, ++round) {
        const uint32_t c1 = T | (1u << b), c2 = T | (2u << b), c3 = T | (3u << b);
        const uint2 n = block_total2(count2(c1, c2, false), count2(c3, 0xFFFFFFFFu, false), round & 1);
        if ((n.y & 0xFFFFu) >= (uint32_t)k) T = c3;
        else if ((n.x >> 16) >= (uint32_t)k) T = c2;
        else if ((n.x & 0xFFFFu) >= (uint32_t)k) T = c1;
      }
      // the last round (15) used buffer 1, so 0 is free
      k_rem = k - (int)(block_total2(count2(T, 0xFFFFFFFFu, true), 0u, 0).x & 0xFFFFu);
    }
  }
  const bool take_all = (k >= n_cand);
  // per thread: a contiguous range of pages so that scans keep page order
  const int per = (n + nthr - 1) / nthr;
  const int lo = min(n, tid * per), hi = min(n, lo + per);
  int ties = 0;
  if (!take_all && k > 0) {
    for (int p = lo; p < min(hi, n_cand); ++p) ties += ((keys[p] & mask) == T);
  }
  int tie_total;
  const int tie_start = block_exclusive_scan(ties, sh_scan, tie_total);
  auto take_of = [&](int p, int& tie_before) -> bool {
    if (p >= n_cand) return keep_newest && p == n - 1;
    if (take_all) return true;
    if (k == 0) return false;
    const uint32_t key = keys[p] & mask;
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

extern "C" argus_status argus_select_workspace_bytes(const argus_geom* g, int32_t batch, int32_t max_pages,
                                                     size_t* bytes) {
  if (!g || !bytes) return fail(ARGUS_E_INVALID, "select: NULL argument");
  if (batch < 0 || max_pages < 0 || g->n_kv_heads <= 0) return fail(ARGUS_E_INVALID, "select: bad sizes");
  *bytes = (size_t)batch * g->n_kv_heads * max_pages * sizeof(uint32_t);
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
  size_t need = (size_t)batch * g->n_kv_heads * max_pages * sizeof(uint32_t);
  if (!ws || ws_bytes < need) return fail(ARGUS_E_WORKSPACE, "select: workspace %zu < %zu", ws_bytes, need);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int G = g->n_q_heads / g->n_kv_heads;
  uint32_t* keys = static_cast<uint32_t*>(ws);
  // pages per CTA: the whole slab in one wave of resident CTAs
  const long long resident = (long long)device_sm_count() * select::kScoreCtasPerSm;
  long long ppc = ((long long)batch * max_pages + resident - 1) / resident;
  ppc = std::max<long long>(8, (ppc + 7) / 8 * 8);
  dim3 grid1((unsigned)((max_pages + ppc - 1) / ppc), batch);
  const size_t sh = (size_t)g->n_kv_heads * g->head_dim * sizeof(float);
  if (sh > 48 * 1024) return fail(ARGUS_E_UNSUPPORTED, "select: n_kv_heads * head_dim too large");
  const uint16_t* ck = static_cast<const uint16_t*>(ckeys);
  const bool bf = (q_dtype == ARGUS_BF16);
  if (g->head_dim == 64) {
    if (bf) select::score_kernel<64, true><<<grid1, select::kScoreThreads, sh, s>>>(g->n_kv_heads, G, max_pages, (int)ppc, q, ck, n_pages, keys);
    else select::score_kernel<64, false><<<grid1, select::kScoreThreads, sh, s>>>(g->n_kv_heads, G, max_pages, (int)ppc, q, ck, n_pages, keys);
  } else {
    if (bf) select::score_kernel<128, true><<<grid1, select::kScoreThreads, sh, s>>>(g->n_kv_heads, G, max_pages, (int)ppc, q, ck, n_pages, keys);
    else select::score_kernel<128, false><<<grid1, select::kScoreThreads, sh, s>>>(g->n_kv_heads, G, max_pages, (int)ppc, q, ck, n_pages, keys);
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
  dim3 grid2(g->n_kv_heads, batch);
  select::topk_kernel<<<grid2, select::kTopkThreads, tsh, s>>>(g->n_kv_heads, max_pages, keys, n_pages, top_k,
                                                               keep_newest, sel_pages, sel_count, sel_width,
                                                               drop_counter, stage);
  return launch_status("argus_select_pages (top-k)");
}
