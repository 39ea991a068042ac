// Host side of the okvq C ABI: configuration checks, the codebook and Hadamard
// signs, device allocation, the decode work partition and the canonical export.
#include <algorithm>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include "okvq_append.h"
#include "okvq_hostio.h"
#include "okvq_internal.h"

using namespace okvq;

struct okvq_cache {
  okvq_config cfg{};
  int S = 0, L = 0, Hq = 0, Hkv = 0, G = 0, bits = 0, M = 0;
  int KG = 0;                   // kernels' group size: G, or 0 for TurboQuant keys
  long long max_tokens = 0, P_max = 0, cap = 0, units = 0;
  PageLayout PL{};
  int num_sms = 0, device = 0;
  // device memory
  uint8_t *pages = nullptr;
  __half *tails = nullptr;      // [2][units][G][D]
  uint8_t *mod = nullptr;       // [S][cap]
  uint32_t *rot_frag = nullptr; // R^T in mma fragment order, fp16 high and residual (see CombineArgs)
  __half *rot_h = nullptr;      // [L*Hkv*M][2][D][D] fp16 high / residual parts of R (append)
  float *signs = nullptr;       // [D]
  uint32_t *err = nullptr;
  float *partials = nullptr;
  int *table = nullptr;         // device work table
  size_t table_bytes = 0;
  long long max_segs = 0;
  int max_cta = 0;
  // host state
  std::vector<long long> len;   // per session
  std::vector<int> tail_sel;    // per session: current tail buffer
  bool dirty = true;
  int ncta = 0, nseg = 0;
  // pinned staging of the work table, two buffers used in turn: a rebuild waits only
  // for the upload two rebuilds back, long finished in an append-decode loop
  void *host_table[2] = {};
  cudaEvent_t table_ev[2] = {};
  bool table_ev_pending[2] = {};
  int table_slot = 0;
  // offsets (bytes) inside the table
  size_t off_segs = 0, off_cta = 0, off_useg = 0, off_ulen = 0, off_utail = 0;
  // codebook
  __half levels16[16];
  __half klev16[16];
  float vthr[15], kthr[15];
  int nlev = 0;
  // eviction and compaction
  std::vector<std::vector<unsigned long long>> dead;   // per session: [P_max] page deletion masks
  unsigned long long *dead_dev = nullptr;              // [S][P_max], the source of the pages' copies
  int *moves_dev = nullptr;                            // [cap / TILE][2] compaction move list
  uint8_t *cscratch = nullptr;                         // compaction gather scratch
  size_t cscratch_bytes = 0;
  // far-memory pseudo tokens
  float *far_partials = nullptr;                       // [units][far_nsplit][MAXGQ][FAR_PARTIAL_FLOATS]
  unsigned char *lut = nullptr;                        // decode level table (LEVEL_TABLE_BYTES)
  __half *q_stage[2] = {}, *out_stage = nullptr;       // device staging of okvq_decode_host
  __half *q_pin = nullptr;                             // its staging of page-locked queries (stage_queries_kernel)
  cudaStream_t copy_stream = nullptr;                  // uploads of okvq_decode_host
  cudaStream_t key_stream = nullptr;                   // the append's key grid, forked from the caller's stream
  cudaEvent_t ev_fork = nullptr, ev_join = nullptr;
  cudaEvent_t ev_in[2] = {}, ev_used[2] = {};          // upload done / staging slot released
  int host_calls = 0;                                  // okvq_decode_host calls that uploaded on copy_stream
  const void *dev_ok[8] = {};                          // device pointers already validated
  int dev_ok_next = 0;
  int far_nsplit = 1;
  // profiling
  bool prof = false;
  std::vector<cudaEvent_t> ev;  // triples per decode call
  int prof_calls = 0;
};

namespace {

constexpr int CTAS_PER_SM = 1;   // the decode kernel holds one 8-warp CTA per SM

uint64_t splitmix64_next(uint64_t &state) {
  state += 0x9E3779B97F4A7C15ull;
  uint64_t z = state;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

double std_normal_pdf(double x) { return std::isfinite(x) ? std::exp(-0.5 * x * x) / std::sqrt(2.0 * M_PI) : 0.0; }
double std_normal_cdf(double x) {
  if (x == INFINITY) return 1.0;
  if (x == -INFINITY) return 0.0;
  return 0.5 * std::erfc(-x / std::sqrt(2.0));
}

// Lloyd-Max quantizer of N(0,1) with n levels: thresholds are midpoints of the
// levels, levels are the conditional means of their cells; iterate to a fixed point.
void lloyd_max(int n, double *lv) {
  for (int j = 0; j < n; ++j) lv[j] = -2.0 + 4.0 * j / (n - 1);
  std::vector<double> th(n + 1), nw(n);
  for (int it = 0; it < 200000; ++it) {
    th[0] = -INFINITY;
    th[n] = INFINITY;
    for (int j = 1; j < n; ++j) th[j] = 0.5 * (lv[j - 1] + lv[j]);
    double delta = 0.0;
    for (int j = 0; j < n; ++j) {
      nw[j] = (std_normal_pdf(th[j]) - std_normal_pdf(th[j + 1])) / (std_normal_cdf(th[j + 1]) - std_normal_cdf(th[j]));
      delta = std::max(delta, std::fabs(nw[j] - lv[j]));
    }
    for (int j = 0; j < n; ++j) lv[j] = nw[j];
    if (delta < 1e-15) break;
  }
}

okvq_status cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return OKVQ_OK;
  if (e == cudaErrorMemoryAllocation) return OKVQ_ENOMEM;
  return OKVQ_ECUDA;
}

#define OKVQ_TRY(expr)                              \
  do {                                              \
    cudaError_t e_ = (expr);                        \
    if (e_ != cudaSuccess) return cuda_status(e_);  \
  } while (0)

// Test hook (okvq_test_fail_alloc): the n-th device allocation from now on fails
// as if the device were out of memory; -1 = off.
std::atomic<long long> g_fail_alloc{-1};

okvq_status alloc_dev(void **p, size_t bytes) {
  long long n = g_fail_alloc.load();
  while (n >= 0 && !g_fail_alloc.compare_exchange_weak(n, n - 1)) {
  }
  if (n == 0) {
    *p = nullptr;
    return OKVQ_ENOMEM;
  }
  cudaError_t e = cudaMalloc(p, bytes ? bytes : 16);
  if (e != cudaSuccess) {
    *p = nullptr;
    return e == cudaErrorMemoryAllocation ? OKVQ_ENOMEM : OKVQ_ECUDA;
  }
  return OKVQ_OK;
}

void release(okvq_cache *h) {
  cudaFree(h->pages);
  cudaFree(h->tails);
  cudaFree(h->mod);
  cudaFree(h->rot_frag);
  cudaFree(h->rot_h);
  cudaFree(h->signs);
  cudaFree(h->err);
  cudaFree(h->partials);
  cudaFree(h->table);
  cudaFree(h->dead_dev);
  cudaFree(h->moves_dev);
  cudaFree(h->cscratch);
  cudaFree(h->far_partials);
  cudaFree(h->lut);
  cudaFree(h->q_stage[0]);
  cudaFree(h->q_stage[1]);
  cudaFree(h->q_pin);
  cudaFree(h->out_stage);
  for (int b = 0; b < 2; ++b) {
    if (h->ev_in[b]) cudaEventDestroy(h->ev_in[b]);
    if (h->ev_used[b]) cudaEventDestroy(h->ev_used[b]);
  }
  if (h->copy_stream) cudaStreamDestroy(h->copy_stream);
  if (h->key_stream) cudaStreamDestroy(h->key_stream);
  if (h->ev_fork) cudaEventDestroy(h->ev_fork);
  if (h->ev_join) cudaEventDestroy(h->ev_join);
  for (int b = 0; b < 2; ++b) {
    if (h->host_table[b]) cudaFreeHost(h->host_table[b]);
    if (h->table_ev[b]) cudaEventDestroy(h->table_ev[b]);
  }
  for (auto e : h->ev) cudaEventDestroy(e);
  delete h;
}

// Split-K partials of okvq_decode_static_scratch: one fixed array per device,
// shared by every call of that entry point (no allocation at call time).
constexpr size_t STATIC_SEG_FLOATS = (size_t)MAXGQ * PARTIAL_FLOATS;
static __device__ __align__(256) float g_static_partials[(size_t)OKVQ_STATIC_SCRATCH_SEGMENTS * STATIC_SEG_FLOATS];

constexpr int MAX_DEVICES = 64;
std::mutex g_static_mu;
float *g_static_addr[MAX_DEVICES] = {};   // device address of g_static_partials, per device

// Look up (once per device, with that device current) the address of the static partials array.
okvq_status static_partials(int device, float **out) {
  if (device < 0 || device >= MAX_DEVICES) return OKVQ_EINVAL;
  std::lock_guard<std::mutex> lock(g_static_mu);
  if (!g_static_addr[device]) {
    int cur = 0;
    if (cudaGetDevice(&cur) != cudaSuccess) return OKVQ_ECUDA;
    if (cur != device && cudaSetDevice(device) != cudaSuccess) return OKVQ_ECUDA;
    void *addr = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&addr, g_static_partials);
    if (cur != device && cudaSetDevice(cur) != cudaSuccess) return OKVQ_ECUDA;
    if (e != cudaSuccess || !addr) return OKVQ_ECUDA;
    g_static_addr[device] = static_cast<float *>(addr);
  }
  *out = g_static_addr[device];
  return OKVQ_OK;
}

// Decode work partition. The flattened (unit, page) list is cut into at most
// max_cta contiguous ranges, one per CTA, and each range into segments at unit
// boundaries. Cost model: a page costs 1, a segment seg_cost more (its query
// rotation, the page ring it starts empty and the cross-warp merge that ends
// it). The smallest per-CTA budget with which a greedy walk covers every page
// is found by bisection (greedy is exact for contiguous splits of an additive
// cost); a segment always holds at least one page. Returns the CTAs used (>= 1
// when there are pages); segs [nseg][4] = unit, first page, end page, 0.
struct SplitPlan {
  int ncta = 0, nseg = 0;
};
SplitPlan plan_split(const long long *pages_u, long long U, int max_cta, int seg_cost, int *segs, int *cta_seg) {
  long long P = 0;
  for (long long u = 0; u < U; ++u) P += pages_u[u];
  SplitPlan r;
  if (P == 0 || max_cta < 1) {
    cta_seg[0] = 0;
    return r;
  }
  const long long sc = std::max(seg_cost, 0);
  // CTAs a budget B needs (emit: also write the segments)
  auto walk = [&](long long B, bool emit) -> long long {
    long long u = 0, p = 0, c = 0;
    int ns = 0;
    while (u < U && pages_u[u] == 0) ++u;
    while (u < U) {
      if (emit) cta_seg[c] = ns;
      long long rem = B;
      while (u < U && rem > sc) {
        const long long take = std::min(pages_u[u] - p, rem - sc);
        if (emit) {
          segs[4 * ns + 0] = (int)u;
          segs[4 * ns + 1] = (int)p;
          segs[4 * ns + 2] = (int)(p + take);
          segs[4 * ns + 3] = 0;
        }
        ++ns;
        rem -= sc + take;
        p += take;
        if (p < pages_u[u]) break;
        p = 0;
        ++u;
        while (u < U && pages_u[u] == 0) ++u;
      }
      ++c;
      if (!emit && c > max_cta) return c;
    }
    if (emit) {
      cta_seg[c] = ns;
      r.nseg = ns;
    }
    return c;
  };
  long long lo = std::max<long long>(sc + 1, (P + max_cta - 1) / max_cta);
  long long hi = P + sc * (U + max_cta) + 1;    // one CTA takes everything
  while (lo < hi) {
    const long long mid = lo + (hi - lo) / 2;
    if (walk(mid, false) <= max_cta) hi = mid;
    else lo = mid + 1;
  }
  r.ncta = (int)walk(lo, true);
  return r;
}

#ifndef OKVQ_SEG_COST
#define OKVQ_SEG_COST 48
#endif
constexpr int SEG_COST_PAGES = OKVQ_SEG_COST;

// Row cost model of a decode CTA. Its W warps take the CTA's pages in turn, so a
// segment of n pages costs ceil(n / W) whole rows of W pages, plus ROW_SEG_COST pages
// for the segment itself (query rotation, the page ring started empty, the merge).
// Measured with 12 warps (2-bit codes, 8 query heads per kv head): a CTA running
// nine 8-page segments takes ~5.1 us per segment, about 24 pages of a loaded CTA's
// time (one row of 12 plus 12).
constexpr int ROW_SEG_COST = 12;

long long row_cost(long long n, int W) { return ROW_SEG_COST + (long long)W * ((n + W - 1) / W); }

// The costliest CTA of a split under the row cost model.
long long split_row_cost(const int *segs, const int *cta_seg, int ncta, int W) {
  long long worst = 0;
  for (int c = 0; c < ncta; ++c) {
    long long t = 0;
    for (int i = cta_seg[c]; i < cta_seg[c + 1]; ++i) t += row_cost(segs[4 * i + 2] - segs[4 * i + 1], W);
    worst = std::max(worst, t);
  }
  return worst;
}

// Row-aligned split: every unit is cut into pieces of R whole rows (R W pages), one
// CTA each, and what is left of each unit (its last pages) goes, costliest first, to
// the least loaded CTA that holds no piece. The smallest R is taken (from the fewest
// rows that could hold every page, trying up to 64 values and at most max_rows, and
// skipping those whose cost fills more than 99.8 % of the CTAs) for which the pieces
// fit in max_cta CTAs and every CTA stays within a piece's cost.
// It uses SMs the contiguous split leaves idle, and it makes every piece whole rows
// (one 512-page unit over two CTAs: pieces of 252 pages, 21 rows, instead of 256
// pages, 22 rows, with the units' 8-page remainders on the idle SMs). Returns the
// CTAs used (0: no R fits); segs [nseg][4] = unit, first page, end page, 0, in CTA
// order; *cost = the costliest CTA's cost.
int plan_rows(const long long *pages_u, long long U, int max_cta, int W, long long max_rows, int *segs, int *cta_seg,
              int *nseg_out, long long *cost) {
  long long P = 0;
  for (long long u = 0; u < U; ++u) P += pages_u[u];
  if (P == 0 || max_cta < 1 || W < 1) return 0;
  std::vector<long long> whole(U);                 // a whole unit as one remainder
  for (long long u = 0; u < U; ++u) whole[u] = pages_u[u] ? row_cost(pages_u[u], W) : 0;
  struct Rest {
    long long cost, unit;
  };
  std::vector<Rest> rest;
  std::vector<std::pair<long long, long long>> placed;   // (bin, unit)
  long long Pmax = 0, total_whole = 0;
  for (long long u = 0; u < U; ++u) {
    Pmax = std::max(Pmax, pages_u[u]);
    total_whole += whole[u];
  }
  bool rest_whole = false;      // `rest` holds every unit whole, sorted (reused while pieces exceed every unit)
  const long long R0 = std::max<long long>(1, (P + (long long)W * max_cta - 1) / ((long long)W * max_cta));
  for (long long R = R0; R <= std::min(max_rows, R0 + 63); ++R) {
    const long long piece = R * W, B = row_cost(piece, W);
    long long main = 0, total = 0;
    if (Pmax < piece) {
      total = total_whole;                  // every unit whole: no pieces
    } else {
      for (long long u = 0; u < U; ++u) {
        const long long p = pages_u[u];
        if (p < piece) {
          total += whole[u];
          continue;
        }
        const long long q = p / piece, r = p - q * piece;
        main += q;
        if (r) total += row_cost(r, W);
      }
    }
    // every CTA holds at most B, and the greedy packing needs some slack: R whose
    // cost fills more than 99.8 % of max_cta CTAs of cost B is not tried
    if (main > max_cta || 1000 * (main * B + total) > 998 * (long long)max_cta * B) continue;
    const long long bins = max_cta - main;
    if (!(Pmax < piece && rest_whole)) {
      rest.clear();
      for (long long u = 0; u < U; ++u) {
        const long long r = pages_u[u] % piece;
        if (r) rest.push_back({pages_u[u] < piece ? whole[u] : row_cost(r, W), u});
      }
      std::stable_sort(rest.begin(), rest.end(), [](const Rest &x, const Rest &y) { return x.cost > y.cost; });
      rest_whole = Pmax < piece;
    }
    if (!rest.empty() && bins == 0) continue;
    // least loaded bin first (ties: lowest index); key = load << 24 | bin
    std::vector<unsigned long long> heap;
    heap.reserve(bins);
    for (long long b = 0; b < bins; ++b) heap.push_back((unsigned long long)b);
    placed.clear();
    bool ok = true;
    for (const Rest &r : rest) {
      const unsigned long long top = heap.front();
      const long long load = (long long)(top >> 24), bin = (long long)(top & 0xFFFFFFull);
      if (load + r.cost > B) {
        ok = false;
        break;
      }
      std::pop_heap(heap.begin(), heap.end(), std::greater<unsigned long long>());
      heap.back() = ((unsigned long long)(load + r.cost) << 24) | (unsigned long long)bin;
      std::push_heap(heap.begin(), heap.end(), std::greater<unsigned long long>());
      placed.push_back({bin, r.unit});
    }
    if (!ok) continue;
    std::sort(placed.begin(), placed.end());
    int ns = 0, c = 0;
    for (long long u = 0; u < U; ++u)
      for (long long k = 0; k < pages_u[u] / piece; ++k) {
        cta_seg[c++] = ns;
        segs[4 * ns + 0] = (int)u;
        segs[4 * ns + 1] = (int)(k * piece);
        segs[4 * ns + 2] = (int)((k + 1) * piece);
        segs[4 * ns + 3] = 0;
        ++ns;
      }
    for (size_t i = 0; i < placed.size(); ++i) {
      if (i == 0 || placed[i].first != placed[i - 1].first) cta_seg[c++] = ns;
      const long long u = placed[i].second;
      segs[4 * ns + 0] = (int)u;
      segs[4 * ns + 1] = (int)(pages_u[u] / piece * piece);
      segs[4 * ns + 2] = (int)pages_u[u];
      segs[4 * ns + 3] = 0;
      ++ns;
    }
    cta_seg[c] = ns;
    *nseg_out = ns;
    *cost = split_row_cost(segs, cta_seg, c, W);
    return c;
  }
  return 0;
}

// Partial slots: a unit's segments get consecutive slots in page order, so the merge
// kernel reads a unit's partials as one range; unit_seg [units + 1] = first slot.
void assign_slots(int *segs, int nseg, long long U, int *unit_seg) {
  std::vector<int> order(nseg);
  for (int i = 0; i < nseg; ++i) order[i] = i;
  std::stable_sort(order.begin(), order.end(), [&](int x, int y) {
    return segs[4 * x] != segs[4 * y] ? segs[4 * x] < segs[4 * y] : segs[4 * x + 1] < segs[4 * y + 1];
  });
  for (int r = 0; r < nseg; ++r) segs[4 * order[r] + 3] = r;
  int sl = 0;
  for (long long uu = 0; uu <= U; ++uu) {
    while (sl < nseg && segs[4 * order[sl]] < uu) ++sl;
    unit_seg[uu] = sl;
  }
}

// The decode's work split: the contiguous split, or the row-aligned one when the row
// cost model puts it at least one row lower.
SplitPlan plan_decode_work(const long long *pages_u, long long U, int max_cta, int W, int *segs, int *cta_seg) {
  SplitPlan sp = plan_split(pages_u, U, max_cta, SEG_COST_PAGES, segs, cta_seg);
  if (sp.ncta == 0) return sp;
  cta_seg[sp.ncta] = sp.nseg;
  const long long contiguous = split_row_cost(segs, cta_seg, sp.ncta, W);
  const long long max_rows = (contiguous - W - ROW_SEG_COST) / W;
  std::vector<int> rsegs(4 * ((size_t)U + max_cta + 1)), rcta(max_cta + 2);
  int rnseg = 0;
  long long rcost = 0;
  const int rn = plan_rows(pages_u, U, max_cta, W, max_rows, rsegs.data(), rcta.data(), &rnseg, &rcost);
  if (rn > 0 && rcost + W <= contiguous) {
    std::copy(rsegs.begin(), rsegs.begin() + 4 * (size_t)rnseg, segs);
    std::copy(rcta.begin(), rcta.begin() + rn + 1, cta_seg);
    sp.ncta = rn;
    sp.nseg = rnseg;
  }
  return sp;
}

// Build the decode work table from the session lengths into pinned buffer `slot`.
void build_table(okvq_cache *h, int slot) {
  const long long U = h->units;
  std::vector<long long> pages_u(U);
  const int LH = h->L * h->Hkv;
  for (long long u = 0; u < U; ++u) {
    long long T = h->len[u / LH];
    pages_u[u] = (T + PAGE - 1) / PAGE;
  }
  char *base = static_cast<char *>(h->host_table[slot]);
  int *segs = reinterpret_cast<int *>(base + h->off_segs);
  int *cta_seg = reinterpret_cast<int *>(base + h->off_cta);
  int *unit_seg = reinterpret_cast<int *>(base + h->off_useg);
  long long *ulen = reinterpret_cast<long long *>(base + h->off_ulen);
  int *utail = reinterpret_cast<int *>(base + h->off_utail);
  for (long long u = 0; u < U; ++u) {
    ulen[u] = h->len[u / LH];
    utail[u] = h->tail_sel[u / LH];
  }
  const SplitPlan sp = plan_decode_work(pages_u.data(), U, h->max_cta, decode_warps(h->bits), segs, cta_seg);
  const int ncta = sp.ncta, nseg = sp.nseg;
  cta_seg[ncta] = nseg;
  assign_slots(segs, nseg, U, unit_seg);
  h->ncta = ncta;
  h->nseg = nseg;
}

constexpr size_t COMPACT_SCRATCH_CAP = 64ull << 20;

// Bytes of one (move, unit) slot of the compaction scratch.
int compaction_stride(const PageLayout &PL, int KG) {
  return (std::max(granule_payload(PL, KG), compaction_granule(KG)) + 15) & ~15;
}

// Ordered-suffix compaction plan over granules ("OmniTide", section 6.2): scan
// suffix starts from the end backward; packing the suffix's non-empty granules in
// order to its start gives length T2; the first start that shortens the
// page-rounded span by min_pages pages is the plan (sg < 0: none).
struct CompactionPlan {
  long long sg = -1, T2 = 0;
  std::vector<int> moves;     // (source granule, destination granule) pairs, ascending
};

CompactionPlan plan_suffix(const std::vector<char> &empty, long long T, int gran, int min_pages) {
  CompactionPlan p;
  const long long ng = (T + gran - 1) / gran, pages0 = (T + PAGE - 1) / PAGE;
  long long kept_tokens = 0;
  for (long long sg = ng - 1; sg >= 0; --sg) {
    if (!empty[sg]) kept_tokens += std::min<long long>(gran, T - sg * gran);
    const long long T2 = sg * gran + kept_tokens;    // only the last granule can be partial
    if (pages0 - (T2 + PAGE - 1) / PAGE >= min_pages) {
      p.sg = sg;
      p.T2 = T2;
      long long dst = sg;
      for (long long j = sg; j < ng; ++j) {
        if (empty[j]) continue;
        if (j != dst) {
          p.moves.push_back((int)j);
          p.moves.push_back((int)dst);
        }
        ++dst;
      }
      return p;
    }
  }
  return p;
}

bool dead_bit(const std::vector<unsigned long long> &w, long long t) { return (w[t >> 6] >> (t & 63)) & 1ull; }
void set_dead_bit(std::vector<unsigned long long> &w, long long t, bool v) {
  if (v) w[t >> 6] |= 1ull << (t & 63);
  else w[t >> 6] &= ~(1ull << (t & 63));
}

// Rewrite the deletion masks (and clear tile masks past the length) of pages
// [p0, p1) of a session from the host copy.
okvq_status push_page_meta(okvq_cache *h, int session, long long p0, long long p1, cudaStream_t s) {
  if (p1 <= p0) return OKVQ_OK;
  unsigned long long *dst = h->dead_dev + (size_t)session * h->P_max + p0;
  // pageable source: staged before the call returns, so the host copy may change afterwards
  OKVQ_TRY(cudaMemcpyAsync(dst, h->dead[session].data() + p0, (size_t)(p1 - p0) * 8, cudaMemcpyHostToDevice, s));
  PageMetaArgs m{};
  m.pages = h->pages;
  m.dead = h->dead_dev + (size_t)session * h->P_max;
  m.LH = h->L * h->Hkv;
  m.session = session;
  m.p0 = p0;
  m.T = h->len[session];
  m.P_max = h->P_max;
  m.PL = h->PL;
  OKVQ_TRY(launch_page_meta(m, (int)(p1 - p0), s));
  return OKVQ_OK;
}

// Upload the work table if the lengths changed, then launch the near-window
// decode, the far-memory kernel (if any) and the merge. seg_limit >= 0: refuse
// (OKVQ_ESCRATCH, nothing launched) a work list with more segments.
okvq_status enqueue_decode(okvq_cache *h, const void *q, void *out, cudaStream_t s, float *partials, long long seg_limit,
                           bool profile, const FarArgs *far) {
  if (h->dirty) {
    const int b = h->table_slot;
    // the staging buffer is free once the upload made from it two rebuilds back has run
    if (h->table_ev_pending[b]) OKVQ_TRY(cudaEventSynchronize(h->table_ev[b]));
    build_table(h, b);
    OKVQ_TRY(cudaMemcpyAsync(h->table, h->host_table[b], h->table_bytes, cudaMemcpyHostToDevice, s));
    OKVQ_TRY(cudaEventRecord(h->table_ev[b], s));
    h->table_ev_pending[b] = true;
    h->table_slot = b ^ 1;
    h->dirty = false;
  }
  if (seg_limit >= 0 && h->nseg > seg_limit) return OKVQ_ESCRATCH;
  const char *tb = reinterpret_cast<const char *>(h->table);
  DecodeArgs a{};
  a.q = static_cast<const __half *>(q);
  a.pages = h->pages;
  a.tails = h->tails;
  a.mod = h->mod;
  a.segs = reinterpret_cast<const int *>(tb + h->off_segs);
  a.cta_seg = reinterpret_cast<const int *>(tb + h->off_cta);
  a.unit_len = reinterpret_cast<const long long *>(tb + h->off_ulen);
  a.unit_tail = reinterpret_cast<const int *>(tb + h->off_utail);
  a.partials = partials;
  a.L = h->L;
  a.Hq = h->Hq;
  a.Hkv = h->Hkv;
  a.M = h->M;
  a.bits = h->bits;
  a.G = h->KG;
  a.P_max = h->P_max;
  a.cap = h->cap;
  a.units = h->units;
  a.lut = h->lut;
  a.signs = h->signs;
  a.err = h->err;
  CombineArgs cb{};
  cb.partials = partials;
  cb.unit_seg = reinterpret_cast<const int *>(tb + h->off_useg);
  cb.rot_frag = reinterpret_cast<const uint4 *>(h->rot_frag);
  cb.err = h->err;
  cb.out = static_cast<__half *>(out);
  cb.L = h->L;
  cb.Hq = h->Hq;
  cb.Hkv = h->Hkv;
  cb.M = h->M;
  cb.units = h->units;
  cb.far = far ? far->partials : nullptr;
  cb.far_split = far ? far->nsplit : 0;
  cudaEvent_t e0 = nullptr, e1 = nullptr, e2 = nullptr;
  if (profile) {
    const size_t need = 3 * (size_t)(h->prof_calls + 1);
    while (h->ev.size() < need) {
      cudaEvent_t ev;
      OKVQ_TRY(cudaEventCreate(&ev));
      h->ev.push_back(ev);
    }
    e0 = h->ev[3 * h->prof_calls];
    e1 = h->ev[3 * h->prof_calls + 1];
    e2 = h->ev[3 * h->prof_calls + 2];
    OKVQ_TRY(cudaEventRecord(e0, s));
  }
  OKVQ_TRY(launch_decode(a, h->ncta, s));
  if (far) OKVQ_TRY(launch_far(*far, s));
  if (profile) OKVQ_TRY(cudaEventRecord(e1, s));
  OKVQ_TRY(launch_combine(cb, s));
  if (profile) {
    OKVQ_TRY(cudaEventRecord(e2, s));
    ++h->prof_calls;
  }
  return OKVQ_OK;
}

// The device address of page-locked, mapped host memory (pinned by cudaHostAlloc
// or registered), else null (pageable memory, or a failed query). Asked on every
// call: a freed pinned buffer's addresses may come back as pageable memory.
void *mapped_host(void *p) {
  cudaPointerAttributes at{};
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    (void)cudaGetLastError();
    return nullptr;
  }
  return at.type == cudaMemoryTypeHost ? at.devicePointer : nullptr;
}

// The decode stages each segment's queries by bulk copy: a 16-byte aligned source.
bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// True for device (or managed) memory of the handle's device; the answer for the
// last few pointers is remembered, so a decode loop on fixed buffers checks once.
bool device_ptr(okvq_cache *h, const void *p) {
  if (!p) return false;
  for (const void *q : h->dev_ok)
    if (q == p) return true;
  cudaPointerAttributes at{};
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    (void)cudaGetLastError();                          // clear the sticky-free error of the query
    return false;
  }
  const bool ok = (at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged) && at.device == h->device;
  if (ok) {
    h->dev_ok[h->dev_ok_next] = p;
    h->dev_ok_next = (h->dev_ok_next + 1) % 8;
  }
  return ok;
}

}  // namespace

extern "C" {

okvq_status okvq_test_fail_alloc(int64_t n) {
  g_fail_alloc.store(n < 0 ? -1 : n);
  return OKVQ_OK;
}

const char *okvq_status_string(okvq_status s) {
  switch (s) {
    case OKVQ_OK: return "ok";
    case OKVQ_EINVAL: return "invalid argument";
    case OKVQ_ENOMEM: return "out of memory";
    case OKVQ_ECAPACITY: return "capacity exceeded";
    case OKVQ_ECUDA: return "CUDA error";
    case OKVQ_ESTATE: return "device error word set";
    case OKVQ_ESCRATCH: return "decode work list exceeds the static scratch array";
  }
  return "unknown status";
}

okvq_status okvq_create(const okvq_config *cfg, void *stream, okvq_cache **out) {
  if (!cfg || !out) return OKVQ_EINVAL;
  *out = nullptr;
  const okvq_config &c = *cfg;
  if (c.num_sessions < 1 || c.num_layers < 1 || c.num_kv_heads < 1 || c.num_q_heads < 1) return OKVQ_EINVAL;
  if (c.num_q_heads % c.num_kv_heads != 0 || c.num_q_heads / c.num_kv_heads > MAXGQ) return OKVQ_EINVAL;
  if (c.head_dim != D) return OKVQ_EINVAL;
  if (c.group_size != 32 && c.group_size != 64) return OKVQ_EINVAL;
  if (c.bits != 2 && c.bits != 4) return OKVQ_EINVAL;
  if (c.num_modalities < 1 || c.num_modalities > MAXM) return OKVQ_EINVAL;
  if (c.key_codec != OKVQ_KEYS_GROUP_RANGE && c.key_codec != OKVQ_KEYS_TURBOQUANT) return OKVQ_EINVAL;
  if (c.max_tokens < 1 || c.max_tokens > (1ll << 31) - PAGE) return OKVQ_EINVAL;   // token indices are 32-bit
  if (!c.value_rot) return OKVQ_EINVAL;
  const int nlev = 1 << c.bits;
  double lv[16];
  if (c.codebook) {
    for (int j = 0; j < nlev; ++j) {
      lv[j] = c.codebook[j];
      if (!std::isfinite(lv[j])) return OKVQ_EINVAL;
      if (j && !(lv[j] > lv[j - 1])) return OKVQ_EINVAL;
    }
  } else {
    lloyd_max(nlev, lv);
  }
  okvq_cache *h = new (std::nothrow) okvq_cache();
  if (!h) return OKVQ_ENOMEM;
  h->cfg = c;
  h->cfg.codebook = nullptr;
  h->cfg.value_rot = nullptr;
  h->S = c.num_sessions;
  h->L = c.num_layers;
  h->Hq = c.num_q_heads;
  h->Hkv = c.num_kv_heads;
  h->G = c.group_size;
  h->bits = c.bits;
  h->M = c.num_modalities;
  h->max_tokens = c.max_tokens;
  h->P_max = (c.max_tokens + PAGE - 1) / PAGE;
  h->cap = h->P_max * PAGE;
  h->units = (long long)h->S * h->L * h->Hkv;
  h->KG = c.key_codec == OKVQ_KEYS_TURBOQUANT ? 0 : h->G;
  h->PL = page_layout(h->bits, h->KG);
  h->len.assign(h->S, 0);
  h->tail_sel.assign(h->S, 0);
  h->dead.assign(h->S, std::vector<unsigned long long>(h->P_max, 0ull));
  // codebook: the fp16-rounded levels define it (values); key levels renormalised to [0, 1]
  h->nlev = nlev;
  double l16[16], k16[16];
  for (int j = 0; j < nlev; ++j) {
    h->levels16[j] = __double2half(lv[j]);
    l16[j] = (double)__half2float(h->levels16[j]);
  }
  for (int j = 0; j < nlev; ++j) {
    h->klev16[j] = __double2half((l16[j] - l16[0]) / (l16[nlev - 1] - l16[0]));
    k16[j] = (double)__half2float(h->klev16[j]);
  }
  for (int j = 0; j + 1 < nlev; ++j) {
    h->vthr[j] = (float)((l16[j] + l16[j + 1]) / 2.0);
    h->kthr[j] = (float)((k16[j] + k16[j + 1]) / 2.0);
  }
  for (int j = nlev - 1; j < 15; ++j) h->vthr[j] = h->kthr[j] = INFINITY;
  for (int j = nlev; j < 16; ++j) h->levels16[j] = h->klev16[j] = __float2half(0.f);

  okvq_status st = OKVQ_OK;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  auto fail = [&](okvq_status e) {
    release(h);
    return e;
  };
  if (cudaGetDevice(&h->device) != cudaSuccess) return fail(OKVQ_ECUDA);
  if (cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, h->device) != cudaSuccess)
    return fail(OKVQ_ECUDA);
  h->max_cta = h->num_sms * CTAS_PER_SM;
  const size_t page_total = (size_t)h->units * h->P_max * h->PL.page_bytes;
  const size_t tails = 2 * (size_t)h->units * h->G * D * sizeof(__half);
  const size_t rot = (size_t)h->L * h->Hkv * h->M * D * D * sizeof(float);
  h->max_segs = (long long)h->max_cta + h->units + 1;
  const size_t partials = (size_t)h->max_segs * MAXGQ * PARTIAL_FLOATS * sizeof(float);
  if ((st = alloc_dev((void **)&h->pages, page_total)) != OKVQ_OK) return fail(st);
  if ((st = alloc_dev((void **)&h->tails, tails)) != OKVQ_OK) return fail(st);
  if ((st = alloc_dev((void **)&h->mod, (size_t)h->S * h->cap)) != OKVQ_OK) return fail(st);
  if ((st = alloc_dev((void **)&h->rot_frag, rot)) != OKVQ_OK) return fail(st);
  const size_t rot_h_bytes = (size_t)h->L * h->Hkv * h->M * 2 * D * D * sizeof(__half);
  if ((st = alloc_dev((void **)&h->rot_h, rot_h_bytes)) != OKVQ_OK) return fail(st);
  if ((st = alloc_dev((void **)&h->signs, D * sizeof(float))) != OKVQ_OK) return fail(st);
  if ((st = alloc_dev((void **)&h->err, sizeof(uint32_t))) != OKVQ_OK) return fail(st);
  if ((st = alloc_dev((void **)&h->partials, partials)) != OKVQ_OK) return fail(st);
  if ((st = alloc_dev((void **)&h->dead_dev, (size_t)h->S * h->P_max * 8)) != OKVQ_OK) return fail(st);
  if ((st = alloc_dev((void **)&h->lut, LEVEL_TABLE_BYTES)) != OKVQ_OK) return fail(st);
  const size_t qo_bytes = (size_t)h->S * h->L * h->Hq * D * sizeof(__half);
  for (int b = 0; b < 2; ++b) {
    if ((st = alloc_dev((void **)&h->q_stage[b], qo_bytes)) != OKVQ_OK) return fail(st);
    if (cudaEventCreateWithFlags(&h->ev_in[b], cudaEventDisableTiming) != cudaSuccess) return fail(OKVQ_ECUDA);
    if (cudaEventCreateWithFlags(&h->ev_used[b], cudaEventDisableTiming) != cudaSuccess) return fail(OKVQ_ECUDA);
  }
  if ((st = alloc_dev((void **)&h->q_pin, qo_bytes)) != OKVQ_OK) return fail(st);
  if ((st = alloc_dev((void **)&h->out_stage, qo_bytes)) != OKVQ_OK) return fail(st);
  if (cudaStreamCreateWithFlags(&h->copy_stream, cudaStreamNonBlocking) != cudaSuccess) return fail(OKVQ_ECUDA);
  if (cudaStreamCreateWithFlags(&h->key_stream, cudaStreamNonBlocking) != cudaSuccess) return fail(OKVQ_ECUDA);
  if (cudaEventCreateWithFlags(&h->ev_fork, cudaEventDisableTiming) != cudaSuccess) return fail(OKVQ_ECUDA);
  if (cudaEventCreateWithFlags(&h->ev_join, cudaEventDisableTiming) != cudaSuccess) return fail(OKVQ_ECUDA);
  // far memory: every unit's pseudo tokens split so that the far grid covers the SMs once
  h->far_nsplit = (int)std::max<long long>(1, (long long)h->num_sms / h->units);
  if ((st = alloc_dev((void **)&h->far_partials,
                      (size_t)h->units * h->far_nsplit * MAXGQ * FAR_PARTIAL_FLOATS * sizeof(float))) != OKVQ_OK)
    return fail(st);
  if ((st = alloc_dev((void **)&h->moves_dev, (size_t)(h->cap / TILE) * 2 * sizeof(int))) != OKVQ_OK) return fail(st);
  {
    // compaction scratch: every granule of a session, or COMPACT_SCRATCH_CAP (larger plans run in batches)
    const int gran = compaction_granule(h->KG);
    const size_t per_move = (size_t)(h->L * h->Hkv + 1) * compaction_stride(h->PL, h->KG);
    h->cscratch_bytes = std::min<size_t>(COMPACT_SCRATCH_CAP, (size_t)(h->cap / gran) * per_move);
    h->cscratch_bytes = std::max(h->cscratch_bytes, per_move);
    if ((st = alloc_dev((void **)&h->cscratch, h->cscratch_bytes)) != OKVQ_OK) return fail(st);
  }
  // work table: segs [max_segs][4] int | cta_seg [max_cta+1] | unit_seg [units+1] | unit_len [units] i64 | unit_tail
  size_t off = 0;
  auto take = [&](size_t bytes) {
    size_t o = off;
    off += (bytes + 15) & ~size_t(15);
    return o;
  };
  h->off_segs = take((size_t)h->max_segs * 4 * sizeof(int));
  h->off_cta = take((size_t)(h->max_cta + 1) * sizeof(int));
  h->off_useg = take((size_t)(h->units + 1) * sizeof(int));
  h->off_ulen = take((size_t)h->units * sizeof(long long));
  h->off_utail = take((size_t)h->units * sizeof(int));
  h->table_bytes = off;
  if ((st = alloc_dev((void **)&h->table, h->table_bytes)) != OKVQ_OK) return fail(st);
  for (int b = 0; b < 2; ++b) {
    if (cudaMallocHost(&h->host_table[b], h->table_bytes) != cudaSuccess) return fail(OKVQ_ENOMEM);
    if (cudaEventCreateWithFlags(&h->table_ev[b], cudaEventDisableTiming) != cudaSuccess) return fail(OKVQ_ECUDA);
  }

  // contents
  if (cudaMemsetAsync(h->pages, 0, page_total, s) != cudaSuccess) return fail(OKVQ_ECUDA);
  if (cudaMemsetAsync(h->tails, 0, tails, s) != cudaSuccess) return fail(OKVQ_ECUDA);
  if (cudaMemsetAsync(h->mod, 0, (size_t)h->S * h->cap, s) != cudaSuccess) return fail(OKVQ_ECUDA);
  if (cudaMemsetAsync(h->err, 0, sizeof(uint32_t), s) != cudaSuccess) return fail(OKVQ_ECUDA);
  if (cudaMemsetAsync(h->dead_dev, 0, (size_t)h->S * h->P_max * 8, s) != cudaSuccess) return fail(OKVQ_ECUDA);
  {
    LutArgs la{};
    la.out = h->lut;
    for (int j = 0; j < 16; ++j) {
      la.klev[j] = h->KG ? h->klev16[j] : h->levels16[j];   // TurboQuant keys use the value levels
      la.vlev[j] = h->levels16[j];
    }
    if (launch_lut(h->bits, la, s) != cudaSuccess) return fail(OKVQ_ECUDA);
  }
  {
    const size_t nmat = (size_t)h->L * h->Hkv * h->M;
    // R as fp16 high + residual parts, row-major [output][channel] (the append
    // kernel's tensor-memory A operand: row o to lane o)
    std::vector<__half> rh(nmat * 2 * D * D);
    for (size_t mtx = 0; mtx < nmat; ++mtx) {
      const float *R = c.value_rot + mtx * D * D;
      __half *H = rh.data() + mtx * 2 * D * D;
      for (int i = 0; i < D; ++i)
        for (int cc = 0; cc < D; ++cc) {
          const float v = R[i * D + cc];
          const __half hi = __float2half_rn(v);
          H[i * D + cc] = hi;
          H[D * D + i * D + cc] = __float2half_rn(v - __half2float(hi));
        }
    }
    // R^T as m16n8k16 A fragments: m-tile mt (16 output channels), k-step ks (16 rows
    // r of the stacked R_m, m = ks / 8), lane (g, t4): a0 = (c = 16mt+g, r = r0..r0+1),
    // a1 = (c+8, r0..), a2 = (c, r0+8..), a3 = (c+8, r0+8..), r0 = 16 (ks%8) + 2 t4;
    // each pair split into an fp16 high part and the fp16 residual
    std::vector<uint32_t> fr(nmat * D * D);
    const int nks = 8 * h->M;
    for (size_t lhm = 0; lhm < (size_t)h->L * h->Hkv; ++lhm)
      for (int mt = 0; mt < 8; ++mt)
        for (int ks = 0; ks < nks; ++ks)
          for (int ln = 0; ln < 32; ++ln)
            for (int i = 0; i < 4; ++i) {
              const int cc = 16 * mt + (ln >> 2) + 8 * (i & 1);
              const int r0 = 16 * (ks % 8) + 2 * (ln & 3) + 8 * (i >> 1);
              const float *Rm = c.value_rot + (lhm * h->M + ks / 8) * D * D;
              const float v0 = Rm[r0 * D + cc], v1 = Rm[(r0 + 1) * D + cc];
              const __half h0 = __float2half_rn(v0), h1 = __float2half_rn(v1);
              const __half l0 = __float2half_rn(v0 - __half2float(h0)), l1 = __float2half_rn(v1 - __half2float(h1));
              const size_t base = (((lhm * 8 + mt) * nks + ks) * 32 + ln) * 8;
              fr[base + i] = (uint32_t)__half_as_ushort(h0) | ((uint32_t)__half_as_ushort(h1) << 16);
              fr[base + 4 + i] = (uint32_t)__half_as_ushort(l0) | ((uint32_t)__half_as_ushort(l1) << 16);
            }
    if (cudaMemcpyAsync(h->rot_frag, fr.data(), rot, cudaMemcpyHostToDevice, s) != cudaSuccess) return fail(OKVQ_ECUDA);
    if (cudaMemcpyAsync(h->rot_h, rh.data(), rot_h_bytes, cudaMemcpyHostToDevice, s) != cudaSuccess)
      return fail(OKVQ_ECUDA);
    uint64_t state = c.hadamard_seed;
    float sg[D];
    for (int w = 0; w < D / 64; ++w) {
      uint64_t z = splitmix64_next(state);
      for (int b = 0; b < 64; ++b) sg[64 * w + b] = ((z >> b) & 1ull) ? -1.f : 1.f;
    }
    if (cudaMemcpyAsync(h->signs, sg, sizeof(sg), cudaMemcpyHostToDevice, s) != cudaSuccess) return fail(OKVQ_ECUDA);
    if (cudaStreamSynchronize(s) != cudaSuccess) return fail(OKVQ_ECUDA);
  }
  *out = h;
  return OKVQ_OK;
}

void okvq_free(okvq_cache *h) {
  if (!h) return;
  cudaDeviceSynchronize();
  release(h);
}

okvq_status okvq_length(const okvq_cache *h, int32_t session, int64_t *tokens) {
  if (!h || !tokens || session < 0 || session >= h->S) return OKVQ_EINVAL;
  *tokens = h->len[session];
  return OKVQ_OK;
}

okvq_status okvq_append_chunk(okvq_cache *h, int32_t session, const void *k, const void *v, const uint8_t *modality,
                              int32_t num_tokens, void *stream) {
  if (!h || session < 0 || session >= h->S || num_tokens < 0) return OKVQ_EINVAL;
  if (num_tokens == 0) return OKVQ_OK;
  if (!device_ptr(h, k) || !device_ptr(h, v) || !device_ptr(h, modality)) return OKVQ_EINVAL;
  if (!aligned16(k) || !aligned16(v)) return OKVQ_EINVAL;
  const long long T0 = h->len[session];
  if (T0 + num_tokens > h->max_tokens) return OKVQ_ECAPACITY;
  AppendArgs a{};
  a.k = static_cast<const __half *>(k);
  a.v = static_cast<const __half *>(v);
  a.mod_in = modality;
  a.n = num_tokens;
  a.T0 = T0;
  a.session = session;
  a.L = h->L;
  a.Hkv = h->Hkv;
  a.M = h->M;
  a.bits = h->bits;
  a.G = h->KG;
  a.P_max = h->P_max;
  a.pages = h->pages;
  const size_t tail_buf = (size_t)h->units * h->G * D;
  a.tail_old = h->tails + (size_t)h->tail_sel[session] * tail_buf;
  a.tail_new = h->tails + (size_t)(1 - h->tail_sel[session]) * tail_buf;
  a.mod = h->mod;
  a.cap = h->cap;
  a.rot_h = h->rot_h;
  a.signs = h->signs;
  a.err = h->err;
  a.page0 = T0 / PAGE;
  a.nlev = h->nlev;
  for (int j = 0; j < 15; ++j) {
    a.vthr[j] = h->vthr[j];
    a.kthr[j] = h->kthr[j];
  }
  const long long last = (T0 + num_tokens - 1) / PAGE;
  const int n_pages = (int)(last - a.page0 + 1);
  // value CTAs: one per SM for short chunks, two per SM (each holds half of the tensor
  // memory) once a unit's chunk spans 24 pages or more (measured: 665-token chunks
  // are faster with one, 2,329-token chunks with two); the key CTAs of the chunk
  // share the SMs with them; at most V_MAX_PPC pages each
  const int upl = h->L * h->Hkv;
  const int per_sm = n_pages >= 24 ? 2 : 1;
  const int cpu = std::max(1, std::min(n_pages, per_sm * h->num_sms / std::max(1, upl)));
  a.vppc = std::min(V_MAX_PPC, (n_pages + cpu - 1) / cpu);
  a.vwide = per_sm == 2 ? 1 : 0;
  cudaError_t e = launch_append(a, n_pages, static_cast<cudaStream_t>(stream), h->key_stream, h->ev_fork, h->ev_join);
  if (e != cudaSuccess) return cuda_status(e);
  h->len[session] = T0 + num_tokens;
  h->tail_sel[session] ^= 1;
  h->dirty = true;
  return OKVQ_OK;
}

okvq_status okvq_decode(okvq_cache *h, const void *q, void *out, void *stream) {
  if (!h || !aligned16(q) || !device_ptr(h, q) || !device_ptr(h, out)) return OKVQ_EINVAL;
  return enqueue_decode(h, q, out, static_cast<cudaStream_t>(stream), h->partials, -1, h->prof, nullptr);
}

okvq_status okvq_decode_host(okvq_cache *h, const void *q_host, void *out_host, void *stream) {
  if (!h || !q_host || !out_host) return OKVQ_EINVAL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t qo_bytes = (size_t)h->S * h->L * h->Hq * D * sizeof(__half);
  // page-locked queries: a kernel on `stream` copies them in (zero-copy reads), so the
  // decode stays a programmatic dependent of the kernel before it and its prologue
  // still overlaps the previous step's merge (stage_queries_kernel)
  const void *q_mapped = aligned16(q_host) ? mapped_host(const_cast<void *>(q_host)) : nullptr;
  const int b = h->host_calls & 1;
  const __half *q_dev = h->q_pin;
  if (q_mapped) {
    OKVQ_TRY(launch_stage_queries(q_mapped, h->q_pin, (long long)(qo_bytes / 16), s));
  } else {
    // pageable queries: the upload runs on the handle's copy stream into one of two
    // staging slots, so it overlaps the decode the previous call left on `stream`; the
    // slot is reused only after the decode two uploads back has read it
    if (h->host_calls >= 2) OKVQ_TRY(cudaStreamWaitEvent(h->copy_stream, h->ev_used[b], 0));
    OKVQ_TRY(cudaMemcpyAsync(h->q_stage[b], q_host, qo_bytes, cudaMemcpyHostToDevice, h->copy_stream));
    OKVQ_TRY(cudaEventRecord(h->ev_in[b], h->copy_stream));
    OKVQ_TRY(cudaStreamWaitEvent(s, h->ev_in[b], 0));
    q_dev = h->q_stage[b];
  }
  // page-locked output: the merge kernel stores into it directly (no copy after the
  // decode); pageable output: device staging, then a copy
  void *out_dev = mapped_host(out_host);
  okvq_status st = enqueue_decode(h, q_dev, out_dev ? out_dev : h->out_stage, s, h->partials, -1, h->prof, nullptr);
  if (st != OKVQ_OK) return st;
  if (!q_mapped) {
    OKVQ_TRY(cudaEventRecord(h->ev_used[b], s));
    ++h->host_calls;
  }
  if (!out_dev) OKVQ_TRY(cudaMemcpyAsync(out_host, h->out_stage, qo_bytes, cudaMemcpyDeviceToHost, s));
  return OKVQ_OK;
}

okvq_status okvq_decode_static_scratch(okvq_cache *h, const void *q, void *out, void *stream) {
  if (!h || !aligned16(q) || !device_ptr(h, q) || !device_ptr(h, out)) return OKVQ_EINVAL;
  float *scratch = nullptr;
  okvq_status st = static_partials(h->device, &scratch);
  if (st != OKVQ_OK) return st;
  // the same launches as okvq_decode, with the partials in the static array
  return enqueue_decode(h, q, out, static_cast<cudaStream_t>(stream), scratch, OKVQ_STATIC_SCRATCH_SEGMENTS, false,
                        nullptr);
}

okvq_status okvq_decode_pseudo(okvq_cache *h, const void *q, const void *far_k, const void *far_v,
                               const float *far_mass, int32_t num_prototypes, int32_t tokens_per_prototype,
                               void *out, void *stream) {
  if (!h || !aligned16(q) || !device_ptr(h, q) || !device_ptr(h, out) || num_prototypes < 0 ||
      tokens_per_prototype < 1)
    return OKVQ_EINVAL;
  const long long n_far = (long long)num_prototypes * tokens_per_prototype;
  if (n_far > (1ll << 30)) return OKVQ_EINVAL;
  if (n_far > 0 && (!device_ptr(h, far_k) || !device_ptr(h, far_v) || !device_ptr(h, far_mass))) return OKVQ_EINVAL;
  if ((reinterpret_cast<uintptr_t>(far_k) | reinterpret_cast<uintptr_t>(far_v)) & 15u) return OKVQ_EINVAL;
  FarArgs f{};
  f.q = static_cast<const __half *>(q);
  f.k = static_cast<const __half *>(far_k);
  f.v = static_cast<const __half *>(far_v);
  f.mass = far_mass;
  f.partials = h->far_partials;
  f.err = h->err;
  f.L = h->L;
  f.Hq = h->Hq;
  f.Hkv = h->Hkv;
  f.n_far = (int)n_far;
  f.per_proto = tokens_per_prototype;
  f.nsplit = h->far_nsplit;
  // tokens per split, a multiple of the tokens one pass of the far kernel's warps takes
  const long long pass = far_pass_tokens();
  f.chunk = (int)(((n_far + h->far_nsplit - 1) / h->far_nsplit + pass - 1) / pass * pass);
  f.units = h->units;
  return enqueue_decode(h, q, out, static_cast<cudaStream_t>(stream), h->partials, -1, h->prof, &f);
}

okvq_status okvq_profile_enable(okvq_cache *h, int enable) {
  if (!h) return OKVQ_EINVAL;
  h->prof = enable != 0;
  h->prof_calls = 0;
  return OKVQ_OK;
}

okvq_status okvq_profile_read(okvq_cache *h, float *split_ms, float *merge_ms, int32_t cap, int32_t *count) {
  if (!h || !count || cap < 0) return OKVQ_EINVAL;
  const int n = std::min<int>(cap, h->prof_calls);
  for (int i = 0; i < n; ++i) {
    OKVQ_TRY(cudaEventSynchronize(h->ev[3 * i + 2]));
    float t1 = 0.f, t2 = 0.f;
    OKVQ_TRY(cudaEventElapsedTime(&t1, h->ev[3 * i], h->ev[3 * i + 1]));
    OKVQ_TRY(cudaEventElapsedTime(&t2, h->ev[3 * i + 1], h->ev[3 * i + 2]));
    if (split_ms) split_ms[i] = t1;
    if (merge_ms) merge_ms[i] = t2;
  }
  *count = n;
  return OKVQ_OK;
}

okvq_status okvq_codebook(const okvq_cache *h, float *levels, float *key_levels) {
  if (!h) return OKVQ_EINVAL;
  for (int j = 0; j < h->nlev; ++j) {
    if (levels) levels[j] = __half2float(h->levels16[j]);
    if (key_levels) key_levels[j] = __half2float(h->klev16[j]);
  }
  return OKVQ_OK;
}

okvq_status okvq_check_errors(okvq_cache *h, void *stream, uint32_t *word) {
  if (!h) return OKVQ_EINVAL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint32_t w = 0;
  OKVQ_TRY(cudaStreamSynchronize(s));
  OKVQ_TRY(cudaMemcpy(&w, h->err, sizeof(w), cudaMemcpyDeviceToHost));
  OKVQ_TRY(cudaMemset(h->err, 0, sizeof(uint32_t)));
  if (word) *word = w;
  return w ? OKVQ_ESTATE : OKVQ_OK;
}

okvq_status okvq_evict(okvq_cache *h, int32_t session, const int64_t *ranges, int32_t num_ranges, void *stream) {
  if (!h || session < 0 || session >= h->S || num_ranges < 0 || (num_ranges > 0 && !ranges)) return OKVQ_EINVAL;
  const long long T = h->len[session];
  long long p0 = -1, p1 = -1;
  for (int i = 0; i < num_ranges; ++i) {
    const long long b = ranges[2 * i], e = ranges[2 * i + 1];
    if (b < 0 || e < b || e > T) return OKVQ_EINVAL;
    if (e == b) continue;
    p0 = p0 < 0 ? b / PAGE : std::min(p0, b / PAGE);
    p1 = std::max(p1, (e - 1) / PAGE + 1);
  }
  if (p0 < 0) return OKVQ_OK;
  for (int i = 0; i < num_ranges; ++i)
    for (long long t = ranges[2 * i]; t < ranges[2 * i + 1]; ++t) set_dead_bit(h->dead[session], t, true);
  return push_page_meta(h, session, p0, p1, static_cast<cudaStream_t>(stream));
}

okvq_status okvq_live_length(const okvq_cache *h, int32_t session, int64_t *tokens) {
  if (!h || !tokens || session < 0 || session >= h->S) return OKVQ_EINVAL;
  const long long T = h->len[session];
  long long dead = 0;
  for (long long p = 0; p < (T + PAGE - 1) / PAGE; ++p) dead += __builtin_popcountll(h->dead[session][p]);
  *tokens = T - dead;
  return OKVQ_OK;
}

okvq_status okvq_compaction_granule(const okvq_cache *h, int32_t *tokens) {
  if (!h || !tokens) return OKVQ_EINVAL;
  *tokens = compaction_granule(h->KG);
  return OKVQ_OK;
}

okvq_status okvq_plan_compaction(const uint8_t *dead, int64_t length, int32_t granule, int32_t min_pages_saved,
                                 int64_t *suffix_begin, int64_t *new_length, int32_t *num_moves) {
  if (length < 0 || (length > 0 && !dead) || min_pages_saved < 1 || !suffix_begin || !new_length || !num_moves)
    return OKVQ_EINVAL;
  if (granule != 16 && granule != 32 && granule != 64) return OKVQ_EINVAL;
  const long long ng = (length + granule - 1) / granule;
  std::vector<char> empty(ng, 1);
  for (long long t = 0; t < length; ++t)
    if (!dead[t]) empty[t / granule] = 0;
  const CompactionPlan p = plan_suffix(empty, length, granule, min_pages_saved);
  *suffix_begin = p.sg < 0 ? -1 : p.sg * granule;
  *new_length = p.sg < 0 ? length : p.T2;
  *num_moves = (int32_t)(p.moves.size() / 2);
  return OKVQ_OK;
}

okvq_status okvq_plan_decode(const int64_t *unit_pages, int64_t units, int32_t max_ctas, int32_t segment_cost,
                             int32_t *segments, int32_t *cta_first, int32_t *num_ctas, int32_t *num_segments) {
  if (units < 0 || (units > 0 && !unit_pages) || max_ctas < 1 || segment_cost < 0 || !segments || !cta_first ||
      !num_ctas || !num_segments)
    return OKVQ_EINVAL;
  if (units > INT32_MAX) return OKVQ_EINVAL;
  std::vector<long long> pages(units);
  for (long long u = 0; u < units; ++u) {
    if (unit_pages[u] < 0 || unit_pages[u] > INT32_MAX) return OKVQ_EINVAL;
    pages[u] = unit_pages[u];
  }
  std::vector<int> segs(4 * (size_t)(units + max_ctas) + 4);
  const SplitPlan sp = plan_split(pages.data(), units, max_ctas, segment_cost, segs.data(), cta_first);
  cta_first[sp.ncta] = sp.nseg;
  for (int i = 0; i < sp.nseg; ++i)
    for (int j = 0; j < 3; ++j) segments[3 * i + j] = segs[4 * i + j];
  *num_ctas = sp.ncta;
  *num_segments = sp.nseg;
  return OKVQ_OK;
}

okvq_status okvq_plan_decode_work(const int64_t *unit_pages, int64_t units, int32_t max_ctas, int32_t bits,
                                  int32_t *segments, int32_t *cta_first, int32_t *unit_first, int32_t *num_ctas,
                                  int32_t *num_segments) {
  if (units < 0 || (units > 0 && !unit_pages) || max_ctas < 1 || (bits != 2 && bits != 4) || !segments ||
      !cta_first || !unit_first || !num_ctas || !num_segments)
    return OKVQ_EINVAL;
  if (units > INT32_MAX) return OKVQ_EINVAL;
  std::vector<long long> pages(units);
  for (long long u = 0; u < units; ++u) {
    if (unit_pages[u] < 0 || unit_pages[u] > INT32_MAX) return OKVQ_EINVAL;
    pages[u] = unit_pages[u];
  }
  std::vector<int> segs(4 * ((size_t)units + max_ctas + 1)), cta(max_ctas + 2);
  const SplitPlan sp = plan_decode_work(pages.data(), units, max_ctas, decode_warps(bits), segs.data(), cta.data());
  cta[sp.ncta] = sp.nseg;
  std::vector<int> useg(units + 1);
  assign_slots(segs.data(), sp.nseg, units, useg.data());
  for (int i = 0; i < 4 * sp.nseg; ++i) segments[i] = segs[i];
  for (int c = 0; c <= sp.ncta; ++c) cta_first[c] = cta[c];
  for (long long u = 0; u <= units; ++u) unit_first[u] = useg[u];
  *num_ctas = sp.ncta;
  *num_segments = sp.nseg;
  return OKVQ_OK;
}

okvq_status okvq_compact(okvq_cache *h, int32_t session, int32_t min_pages_saved, int64_t *new_length,
                         int32_t *moved_granules, void *stream) {
  if (!h || session < 0 || session >= h->S || min_pages_saved < 1) return OKVQ_EINVAL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const long long T = h->len[session];
  const int gran = compaction_granule(h->KG);
  const long long ng = (T + gran - 1) / gran;
  std::vector<char> empty(ng, 1);
  for (long long t = 0; t < T; ++t)
    if (!dead_bit(h->dead[session], t)) empty[t / gran] = 0;
  const CompactionPlan p = plan_suffix(empty, T, gran, min_pages_saved);
  const int n = (int)(p.moves.size() / 2);
  if (new_length) *new_length = p.sg < 0 ? T : p.T2;
  if (moved_granules) *moved_granules = n;
  if (p.sg < 0) return OKVQ_OK;
  const int LH = h->L * h->Hkv;
  if (n > 0) {
    const int stride = compaction_stride(h->PL, h->KG);
    const size_t per_move = (size_t)(LH + 1) * stride;
    const int batch = (int)std::min<size_t>((size_t)n, h->cscratch_bytes / per_move);
    OKVQ_TRY(cudaMemcpyAsync(h->moves_dev, p.moves.data(), p.moves.size() * sizeof(int), cudaMemcpyHostToDevice, s));
    MoveArgs m{};
    m.pages = h->pages;
    m.mod = h->mod;
    m.scratch = h->cscratch;
    m.LH = LH;
    m.KG = h->KG;
    m.session = session;
    m.stride = stride;
    m.P_max = h->P_max;
    m.cap = h->cap;
    m.PL = h->PL;
    // every destination of a batch lies below every source of the later batches,
    // and a batch's sources are all gathered before any of its destinations is written
    for (int k0 = 0; k0 < n; k0 += batch) {
      m.moves = h->moves_dev + 2 * k0;
      m.n = std::min(batch, n - k0);
      m.scatter = 0;
      OKVQ_TRY(launch_move(m, s));
      m.scatter = 1;
      OKVQ_TRY(launch_move(m, s));
    }
  }
  // the host copy of the deletion masks follows the moves
  std::vector<unsigned long long> &w = h->dead[session];
  for (int k = 0; k < n; ++k) {
    const long long src = (long long)p.moves[2 * k] * gran, dst = (long long)p.moves[2 * k + 1] * gran;
    const long long cnt = std::min<long long>(gran, T - src);
    for (long long i = 0; i < cnt; ++i) set_dead_bit(w, dst + i, dead_bit(w, src + i));
  }
  for (long long t = p.T2; t < T; ++t) set_dead_bit(w, t, false);
  h->len[session] = p.T2;
  h->dirty = true;
  return push_page_meta(h, session, (p.sg * gran) / PAGE, (T + PAGE - 1) / PAGE, s);
}

okvq_status okvq_export_state(okvq_cache *h, int32_t session, void *host_buf, size_t *bytes) {
  if (!h || !bytes || session < 0 || session >= h->S) return OKVQ_EINVAL;
  const long long T = h->len[session];
  const int G = h->G, bits = h->bits;
  const bool turbo = h->KG == 0;
  const long long Tf = turbo ? T : (T / G) * G;
  const int B = D * bits / 8;
  const long long LH = (long long)h->L * h->Hkv;
  // TurboQuant keys: knorm [LH][T] fp16 in the kstats slot, no tail
  const size_t n_kc = (size_t)LH * Tf * B,
               n_ks = turbo ? (size_t)LH * T * 2 : (size_t)LH * (Tf / G) * 2 * D * 2,
               n_kt = (size_t)LH * (T - Tf) * D * 2, n_vc = (size_t)LH * T * B, n_vn = (size_t)LH * T * 2,
               n_md = (size_t)T, n_dd = (size_t)LH * T;
  const size_t need = n_kc + n_ks + n_kt + n_vc + n_vn + n_md + n_dd;
  if (!host_buf) {
    *bytes = need;
    return OKVQ_OK;
  }
  if (*bytes < need) return OKVQ_EINVAL;
  *bytes = need;
  OKVQ_TRY(cudaDeviceSynchronize());
  uint8_t *out = static_cast<uint8_t *>(host_buf);
  uint8_t *o_kc = out, *o_ks = o_kc + n_kc, *o_kt = o_ks + n_ks, *o_vc = o_kt + n_kt, *o_vn = o_vc + n_vc,
          *o_md = o_vn + n_vn, *o_dd = o_md + n_md;
  std::memset(out, 0, need);
  const long long npages = (T + PAGE - 1) / PAGE;
  const PageLayout PL = h->PL;
  std::vector<uint8_t> pg((size_t)npages * PL.page_bytes);
  std::vector<__half> tail((size_t)G * D);
  // where code (tok in tile, channel) sits: lane chunk and bit, for K and V layouts
  std::vector<int> kpos(TILE * D), vpos(TILE * D);
  for (int lane = 0; lane < 32; ++lane)
    for (int j = 0; j < 32; ++j)
      for (int e = 0; e < 2; ++e) {
        int tok, ch;
        k_pair_coords(lane, j, e, tok, ch);
        kpos[tok * D + ch] = lane * PL.lane_bytes * 8 + k_code_bit(bits, j, e);
        v_pair_coords(lane, j, e, tok, ch);
        vpos[tok * D + ch] = lane * PL.lane_bytes * 8 + v_code_bit(bits, j, e);
      }
  int inv_stat[D];
  for (int p = 0; p < D; ++p) inv_stat[stat_channel(p)] = p;
  const uint32_t mask = (1u << bits) - 1u;
  for (long long lh = 0; lh < LH; ++lh) {
    const long long unit = (long long)session * LH + lh;
    if (npages)
      OKVQ_TRY(cudaMemcpy(pg.data(), h->pages + (unit * h->P_max) * PL.page_bytes, (size_t)npages * PL.page_bytes,
                          cudaMemcpyDeviceToHost));
    for (long long t = 0; t < T; ++t) {
      const uint8_t *p = pg.data() + (t / PAGE) * PL.page_bytes;
      const int tt = (int)(t % PAGE), tile = tt / TILE, r = tt % TILE;
      for (int ch = 0; ch < D; ++ch) {
        int vb = vpos[r * D + ch];
        uint32_t vc = (p[PL.off_v + tile * PL.tile_bytes + vb / 8] >> (vb % 8)) & mask;
        o_vc[(lh * T + t) * B + ch * bits / 8] |= (uint8_t)(vc << ((ch * bits) % 8));
        if (t < Tf) {
          int kbp = kpos[r * D + ch];
          uint32_t kc = (p[tile * PL.tile_bytes + kbp / 8] >> (kbp % 8)) & mask;
          o_kc[(lh * Tf + t) * B + ch * bits / 8] |= (uint8_t)(kc << ((ch * bits) % 8));
        }
      }
      std::memcpy(o_vn + (lh * T + t) * 2, p + PL.off_norm + tt * 2, 2);
      unsigned long long dw;
      std::memcpy(&dw, p + PL.off_tmask + DEAD_OFF, 8);
      o_dd[lh * T + t] = (uint8_t)((dw >> tt) & 1ull);
    }
    if (turbo) {
      for (long long t = 0; t < T; ++t)
        std::memcpy(o_ks + (lh * T + t) * 2, pg.data() + (t / PAGE) * PL.page_bytes + PL.off_stats + (t % PAGE) * 2, 2);
    }
    for (long long gi = 0; !turbo && gi < Tf / G; ++gi) {
      const uint8_t *p = pg.data() + ((gi * G) / PAGE) * PL.page_bytes + PL.off_stats + ((gi * G) % PAGE) / G * 2 * D * 2;
      const __half *st = reinterpret_cast<const __half *>(p);
      __half *dst = reinterpret_cast<__half *>(o_ks) + (lh * (Tf / G) + gi) * 2 * D;
      for (int ch = 0; ch < D; ++ch) {
        dst[ch] = st[inv_stat[ch]];
        dst[D + ch] = st[D + inv_stat[ch]];
      }
    }
    if (T > Tf) {
      const __half *src = h->tails + ((size_t)h->tail_sel[session] * h->units + unit) * G * D;
      OKVQ_TRY(cudaMemcpy(tail.data(), src, (size_t)(T - Tf) * D * 2, cudaMemcpyDeviceToHost));
      std::memcpy(o_kt + (size_t)lh * (T - Tf) * D * 2, tail.data(), (size_t)(T - Tf) * D * 2);
    }
  }
  if (T) OKVQ_TRY(cudaMemcpy(o_md, h->mod + (size_t)session * h->cap, (size_t)T, cudaMemcpyDeviceToHost));
  return OKVQ_OK;
}

}  // extern "C"
