// Eviction and compaction of the packed cache ("OmniTide: Co-Designing
// Algorithms and Systems for Efficient On-Device Omni-LLM Streaming", section
// 5.2 Applying the retention plan: deleted ranges leave holes and survivors keep
// their slots; section 6.2 Selective and efficient KV migration: the
// ordered-suffix mode packs the surviving entries of a suffix, and on CUDA the
// sources are gathered into scratch space before the destinations are written,
// so that no write lands on a source another move still needs).
//
// move_kernel      - one CTA per (move, layer x kv head) plus one per move for the
//                    session's modality ids: copies one granule's bytes between its
//                    page slot and the scratch slot (gather or scatter).
// page_meta_kernel - one CTA per (page, layer x kv head): writes the page's
//                    deletion mask from the session's mask array and clears the
//                    tile modality masks of tiles at or past the session length.
#include "okvq_internal.h"

namespace okvq {

namespace {

constexpr int MOVE_THREADS = 128;

// Copy `bytes` (a multiple of 16, both addresses 16-byte aligned) with 16-byte accesses.
__device__ __forceinline__ void copy16(uint8_t *dst, const uint8_t *src, int bytes) {
  for (int i = threadIdx.x; i < bytes / 16; i += MOVE_THREADS)
    reinterpret_cast<uint4 *>(dst)[i] = reinterpret_cast<const uint4 *>(src)[i];
}

__global__ void __launch_bounds__(MOVE_THREADS) move_kernel(const MoveArgs a) {
  const int k = blockIdx.x, lh = blockIdx.y;
  const int gran = compaction_granule(a.KG), nt = gran / TILE;
  const long long gi = a.moves[2 * k + (a.scatter ? 1 : 0)];     // the page-side granule
  const long long tok = gi * gran;
  uint8_t *slot = a.scratch + ((long long)k * (a.LH + 1) + lh) * a.stride;
  if (lh == a.LH) {                                              // modality ids (gran is a multiple of 16)
    uint8_t *m = a.mod + (long long)a.session * a.cap + tok;
    if (a.scatter) copy16(m, slot, gran);
    else copy16(slot, m, gran);
    return;
  }
  const PageLayout &PL = a.PL;
  const long long unit = (long long)a.session * a.LH + lh;
  uint8_t *pg = a.pages + (unit * a.P_max + tok / PAGE) * (long long)PL.page_bytes;
  const int tin = (int)(tok % PAGE), tb = tin / TILE;
  // the granule's pieces inside the page, in scratch order
  const int off[4] = {tb * PL.tile_bytes, PL.off_v + tb * PL.tile_bytes, PL.off_norm + 2 * tin,
                      PL.off_stats + (a.KG ? (tin / a.KG) * 2 * D * 2 : 2 * tin)};
  const int len[4] = {nt * PL.tile_bytes, nt * PL.tile_bytes, 2 * gran, a.KG ? 2 * D * 2 : 2 * gran};
  int so = 0;
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    if (a.scatter) copy16(pg + off[p], slot + so, len[p]);
    else copy16(slot + so, pg + off[p], len[p]);
    so += len[p];
  }
  if (threadIdx.x < nt) {                                        // tile modality masks
    if (a.scatter) pg[PL.off_tmask + tb + threadIdx.x] = slot[so + threadIdx.x];
    else slot[so + threadIdx.x] = pg[PL.off_tmask + tb + threadIdx.x];
  }
}

__global__ void page_meta_kernel(const PageMetaArgs a) {
  const long long page = a.p0 + blockIdx.x;
  const int lh = blockIdx.y;
  const long long unit = (long long)a.session * a.LH + lh;
  uint8_t *pg = a.pages + (unit * a.P_max + page) * (long long)a.PL.page_bytes;
  if (threadIdx.x == 0)
    *reinterpret_cast<unsigned long long *>(pg + a.PL.off_tmask + DEAD_OFF) = a.dead[page];
  if (threadIdx.x < PAGE / TILE && page * PAGE + TILE * threadIdx.x >= a.T) pg[a.PL.off_tmask + threadIdx.x] = 0;
}

}  // namespace

cudaError_t launch_move(const MoveArgs &a, cudaStream_t s) {
  if (a.n <= 0) return cudaSuccess;
  move_kernel<<<dim3((unsigned)a.n, (unsigned)(a.LH + 1)), MOVE_THREADS, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_page_meta(const PageMetaArgs &a, int n_pages, cudaStream_t s) {
  if (n_pages <= 0) return cudaSuccess;
  page_meta_kernel<<<dim3((unsigned)n_pages, (unsigned)a.LH), 32, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace okvq
