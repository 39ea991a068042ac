// Eviction and compaction of the packed cache ("OmniTide: Co-Designing
// Algorithms and Systems for Efficient On-Device Omni-LLM Streaming", section
// 5.2 Applying the retention plan: deleted ranges leave holes and survivors keep
// their slots; section 6.2 Selective and efficient KV migration: the
// ordered-suffix mode packs the surviving entries of a suffix, and on CUDA the
// sources are gathered into scratch space before the destinations are written,
// so that no write lands on a source another move still needs).
//
// move_kernel      - one CTA per (move, 8 layer x kv head slots; the last group
//                    also carries the session's modality ids): copies one granule's
//                    bytes between its page slots and the scratch slots (gather or
//                    scatter).
// page_meta_kernel - one thread per (page, layer x kv head), flat grid: writes the
//                    page's deletion mask from the session's mask array and
//                    clears the tile modality masks of tiles at or past the
//                    session length.
#include "okvq_internal.h"

namespace okvq {

namespace {

constexpr int MOVE_THREADS = 256;
constexpr int MOVE_UNITS = 8;          // (layer, kv head) slots per CTA

// Copy `bytes` (a multiple of 16, both addresses 16-byte aligned) with 16-byte accesses.
__device__ __forceinline__ void copy16(uint8_t *dst, const uint8_t *src, int bytes) {
  for (int i = threadIdx.x; i < bytes / 16; i += MOVE_THREADS)
    reinterpret_cast<uint4 *>(dst)[i] = reinterpret_cast<const uint4 *>(src)[i];
}

// One CTA per (move, group of MOVE_UNITS (layer, kv head) slots): the slots'
// pieces form one list of 16-byte words, spread over all the CTA's threads.
__global__ void __launch_bounds__(MOVE_THREADS) move_kernel(const MoveArgs a) {
  const int k = blockIdx.x;
  const int gran = compaction_granule(a.KG), nt = gran / TILE;
  const long long gi = a.moves[2 * k + (a.scatter ? 1 : 0)];     // the page-side granule
  const long long tok = gi * gran;
  const PageLayout &PL = a.PL;
  const int tin = (int)(tok % PAGE), tb = tin / TILE;
  // the granule's pieces inside a page, in scratch order (lengths in 16-byte words)
  const int off[4] = {tb * PL.tile_bytes, PL.off_v + tb * PL.tile_bytes, PL.off_norm + 2 * tin,
                      PL.off_stats + (a.KG ? (tin / a.KG) * 2 * D * 2 : 2 * tin)};
  const int len[4] = {nt * PL.tile_bytes / 16, nt * PL.tile_bytes / 16, 2 * gran / 16,
                      (a.KG ? 2 * D * 2 : 2 * gran) / 16};
  const int per = len[0] + len[1] + len[2] + len[3];
  const int lh0 = blockIdx.y * MOVE_UNITS, lh1 = min(a.LH, lh0 + MOVE_UNITS);
  uint8_t *scr = a.scratch + (long long)k * (a.LH + 1) * a.stride;
  for (int idx = threadIdx.x; idx < (lh1 - lh0) * per; idx += MOVE_THREADS) {
    const int lh = lh0 + idx / per, w = idx % per;
    // piece of word w: cumulative bounds, no indexed arrays (they would live in local memory)
    const int c1 = len[0], c2 = c1 + len[1], c3 = c2 + len[2];
    const int so = w >= c3 ? c3 : w >= c2 ? c2 : w >= c1 ? c1 : 0;
    const int po = w >= c3 ? off[3] : w >= c2 ? off[2] : w >= c1 ? off[1] : off[0];
    const long long unit = (long long)a.session * a.LH + lh;
    uint4 *pg = reinterpret_cast<uint4 *>(a.pages + (unit * a.P_max + tok / PAGE) * (long long)PL.page_bytes + po) +
                (w - so);
    uint4 *sl = reinterpret_cast<uint4 *>(scr + (long long)lh * a.stride) + w;
    if (a.scatter) *pg = *sl;
    else *sl = *pg;
  }
  for (int idx = threadIdx.x; idx < (lh1 - lh0) * nt; idx += MOVE_THREADS) {   // tile modality masks
    const int lh = lh0 + idx / nt, j = idx % nt;
    const long long unit = (long long)a.session * a.LH + lh;
    uint8_t *pg = a.pages + (unit * a.P_max + tok / PAGE) * (long long)PL.page_bytes + PL.off_tmask + tb + j;
    uint8_t *sl = scr + (long long)lh * a.stride + 16 * per + j;
    if (a.scatter) *pg = *sl;
    else *sl = *pg;
  }
  if (a.LH >= lh0 && a.LH < lh0 + MOVE_UNITS) {                  // modality ids (gran is a multiple of 16)
    uint8_t *m = a.mod + (long long)a.session * a.cap + tok;
    uint8_t *sl = scr + (long long)a.LH * a.stride;
    if (a.scatter) copy16(m, sl, gran);
    else copy16(sl, m, gran);
  }
}

constexpr int META_THREADS = 256;

__global__ void __launch_bounds__(META_THREADS) page_meta_kernel(const PageMetaArgs a, long long n) {
  const long long i = (long long)blockIdx.x * META_THREADS + threadIdx.x;
  if (i >= n) return;
  const long long page = a.p0 + i / a.LH;       // consecutive threads: the units of one page
  const int lh = (int)(i % a.LH);
  const long long unit = (long long)a.session * a.LH + lh;
  uint8_t *pg = a.pages + (unit * a.P_max + page) * (long long)a.PL.page_bytes;
  *reinterpret_cast<unsigned long long *>(pg + a.PL.off_tmask + DEAD_OFF) = a.dead[page];
#pragma unroll
  for (int t = 0; t < PAGE / TILE; ++t)
    if (page * PAGE + TILE * t >= a.T) pg[a.PL.off_tmask + t] = 0;
}

}  // namespace

cudaError_t launch_move(const MoveArgs &a, cudaStream_t s) {
  if (a.n <= 0) return cudaSuccess;
  move_kernel<<<dim3((unsigned)a.n, (unsigned)((a.LH + 1 + MOVE_UNITS - 1) / MOVE_UNITS)), MOVE_THREADS, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_page_meta(const PageMetaArgs &a, int n_pages, cudaStream_t s) {
  if (n_pages <= 0) return cudaSuccess;
  const long long n = (long long)n_pages * a.LH;
  page_meta_kernel<<<(unsigned)((n + META_THREADS - 1) / META_THREADS), META_THREADS, 0, s>>>(a, n);
  return cudaGetLastError();
}

}  // namespace okvq
