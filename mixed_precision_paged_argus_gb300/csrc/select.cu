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
// (D bf16 per page and head); CTAs tile (batch row, page range), lanes read 16
// bytes of a compressed key each and reduce within the head's lanes; the
// G-query sum is formed once per CTA in shared memory.  (2) top-k: one CTA per
// (batch row, KV head) radix-selects the k-th largest score over the L2-resident
// score row (four 8-bit passes with shared-memory histograms), then compacts
// the chosen pages in ascending order with block-wide prefix sums.
#include <algorithm>

#include "common.cuh"

namespace argus {
namespace select {

constexpr int kScoreThreads = 256;
constexpr int kPagesPerCta = 64;
constexpr int kTopkThreads = 512;

template <int D, bool QBF16>
__global__ void __launch_bounds__(kScoreThreads) score_kernel(int Hkv, int G, int max_pages, const void* q,
                                                              const uint16_t* ckeys, const int32_t* n_pages,
                                                              float* scores) {
  extern __shared__ float qsum[];  // [Hkv][D]
  const int b = blockIdx.y;
  const int p0 = blockIdx.x * kPagesPerCta;
  const int Hq = Hkv * G;
  int n = n_pages[b];
  n = max(0, min(n, max_pages));
  if (p0 >= n) return;
  const uint16_t* qb = static_cast<const uint16_t*>(q) + (size_t)b * Hq * D;
  for (int idx = threadIdx.x; idx < Hkv * D; idx += blockDim.x) {
    const int h = idx / D, d = idx - h * D;
    float s = 0.f;
    for (int g = 0; g < G; ++g) {
      const uint16_t bits = qb[(size_t)(h * G + g) * D + d];
      s += QBF16 ? __uint_as_float((uint32_t)bits << 16) : __half2float(__ushort_as_half(bits));
    }
    qsum[idx] = s;
  }
  __syncthreads();
  constexpr int LPH = D / 8;  // lanes per (page, head) row
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int rows_per_warp = 32 / LPH;
  const int sub = lane / LPH, li = lane % LPH;
  const int p_end = min(n, p0 + kPagesPerCta);
  const int n_rows = (p_end - p0) * Hkv;
  for (int row = warp * rows_per_warp + sub; row - sub < n_rows; row += (blockDim.x / 32) * rows_per_warp) {
    float s = 0.f;
    const bool live = row < n_rows;
    int p = 0, h = 0;
    if (live) {
      p = p0 + row / Hkv;
      h = row % Hkv;
      const uint4 x = *reinterpret_cast<const uint4*>(ckeys + (((size_t)b * max_pages + p) * Hkv + h) * D + 8 * li);
      const uint32_t w[4] = {x.x, x.y, x.z, x.w};
      const float* qs = qsum + h * D + 8 * li;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float k = __uint_as_float(((w[e / 2] >> (16 * (e & 1))) & 0xFFFFu) << 16);
        s = fmaf(k, qs[e], s);
      }
    }
#pragma unroll
    for (int o = 1; o < LPH; o <<= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (live && li == 0) scores[((size_t)b * Hkv + h) * max_pages + p] = s;
  }
}

__device__ __forceinline__ uint32_t order_key(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
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

__global__ void __launch_bounds__(kTopkThreads) topk_kernel(int Hkv, int max_pages, const float* scores,
                                                            const int32_t* n_pages, int top_k, int keep_newest,
                                                            int32_t* sel_pages, int32_t* sel_count, int width,
                                                            uint32_t* drops) {
  __shared__ int hist[256];
  __shared__ int sh_scan[32];
  __shared__ int sh_sel[2];
  const int h = blockIdx.x, b = blockIdx.y;
  const int tid = threadIdx.x, nthr = blockDim.x;
  int n = n_pages[b];
  const int n_raw = n;
  n = max(0, min(n, max_pages));
  int32_t* out = sel_pages + ((size_t)b * Hkv + h) * width;
  const float* sc = scores + ((size_t)b * Hkv + h) * max_pages;
  uint32_t dropped = 0;
  if (n_raw > max_pages && tid == 0 && h == 0) dropped += (uint32_t)(n_raw - max_pages);
  const int n_cand = (n > 0) ? (keep_newest ? n - 1 : n) : 0;
  const int room = width - ((keep_newest && n > 0) ? 1 : 0);
  const int k_want = min(top_k, n_cand);
  const int k = max(0, min(k_want, room));
  if (tid == 0) dropped += (uint32_t)(k_want - k);

  // threshold T = k-th largest key; take all > T and the first k_rem equal to T
  uint32_t T = 0u;
  int k_rem = 0;
  if (k > 0 && k < n_cand) {
    uint32_t prefix = 0u, mask = 0u;
    int need = k;
    for (int pass = 0; pass < 4; ++pass) {
      const int shift = 24 - 8 * pass;
      for (int i = tid; i < 256; i += nthr) hist[i] = 0;
      __syncthreads();
      for (int p = tid; p < n_cand; p += nthr) {
        const uint32_t key = order_key(sc[p]);
        if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 255], 1);
      }
      __syncthreads();
      if (tid == 0) {
        int acc = 0, dsel = 0;
        for (int d = 255; d >= 0; --d) {
          if (acc + hist[d] >= need) {
            dsel = d;
            break;
          }
          acc += hist[d];
        }
        sh_sel[0] = dsel;
        sh_sel[1] = need - acc;
      }
      __syncthreads();
      prefix |= (uint32_t)sh_sel[0] << shift;
      mask |= 255u << shift;
      need = sh_sel[1];
      __syncthreads();
    }
    T = prefix;
    k_rem = need;
  }
  const bool take_all = (k >= n_cand);
  // per thread: a contiguous range of pages so that scans keep page order
  const int per = (n + nthr - 1) / nthr;
  const int lo = min(n, tid * per), hi = min(n, lo + per);
  int ties = 0;
  if (!take_all && k > 0) {
    for (int p = lo; p < min(hi, n_cand); ++p) ties += (order_key(sc[p]) == T);
  }
  int tie_total;
  int tie_before = block_exclusive_scan(ties, sh_scan, tie_total);
  int mine = 0;
  for (int p = lo; p < hi; ++p) {
    bool take;
    if (p >= n_cand) take = keep_newest && p == n - 1;
    else if (take_all) take = true;
    else if (k == 0) take = false;
    else {
      const uint32_t key = order_key(sc[p]);
      if (key > T) take = true;
      else if (key == T) take = (tie_before++ < k_rem);
      else take = false;
    }
    mine += take;
  }
  int total;
  int pos = block_exclusive_scan(mine, sh_scan, total);
  tie_before = block_exclusive_scan(ties, sh_scan, tie_total);
  for (int p = lo; p < hi; ++p) {
    bool take;
    if (p >= n_cand) take = keep_newest && p == n - 1;
    else if (take_all) take = true;
    else if (k == 0) take = false;
    else {
      const uint32_t key = order_key(sc[p]);
      if (key > T) take = true;
      else if (key == T) take = (tie_before++ < k_rem);
      else take = false;
    }
    if (take && pos < width) out[pos++] = p;
  }
  __syncthreads();
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
  *bytes = (size_t)batch * g->n_kv_heads * max_pages * sizeof(float);
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
  if (batch == 0) return ARGUS_OK;
  if (!q || !ckeys || !n_pages || !sel_pages || !sel_count)
    return fail(ARGUS_E_INVALID, "select: NULL pointer");
  if (reinterpret_cast<uintptr_t>(ckeys) & 15) return fail(ARGUS_E_INVALID, "select: ckeys not 16-byte aligned");
  size_t need = (size_t)batch * g->n_kv_heads * max_pages * sizeof(float);
  if (!ws || ws_bytes < need) return fail(ARGUS_E_WORKSPACE, "select: workspace %zu < %zu", ws_bytes, need);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int G = g->n_q_heads / g->n_kv_heads;
  float* scores = static_cast<float*>(ws);
  dim3 grid1((max_pages + select::kPagesPerCta - 1) / select::kPagesPerCta, batch);
  const size_t sh = (size_t)g->n_kv_heads * g->head_dim * sizeof(float);
  if (sh > 48 * 1024) return fail(ARGUS_E_UNSUPPORTED, "select: n_kv_heads * head_dim too large");
  const uint16_t* ck = static_cast<const uint16_t*>(ckeys);
  const bool bf = (q_dtype == ARGUS_BF16);
  if (g->head_dim == 64) {
    if (bf) select::score_kernel<64, true><<<grid1, select::kScoreThreads, sh, s>>>(g->n_kv_heads, G, max_pages, q, ck, n_pages, scores);
    else select::score_kernel<64, false><<<grid1, select::kScoreThreads, sh, s>>>(g->n_kv_heads, G, max_pages, q, ck, n_pages, scores);
  } else {
    if (bf) select::score_kernel<128, true><<<grid1, select::kScoreThreads, sh, s>>>(g->n_kv_heads, G, max_pages, q, ck, n_pages, scores);
    else select::score_kernel<128, false><<<grid1, select::kScoreThreads, sh, s>>>(g->n_kv_heads, G, max_pages, q, ck, n_pages, scores);
  }
  argus_status st = launch_status("argus_select_pages (score)");
  if (st != ARGUS_OK) return st;
  dim3 grid2(g->n_kv_heads, batch);
  select::topk_kernel<<<grid2, select::kTopkThreads, 0, s>>>(g->n_kv_heads, max_pages, scores, n_pages, top_k,
                                                             keep_newest, sel_pages, sel_count, sel_width,
                                                             drop_counter);
  return launch_status("argus_select_pages (top-k)");
}
