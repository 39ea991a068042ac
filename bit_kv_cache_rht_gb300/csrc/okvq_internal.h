// Internal definitions of libokvq: device layout of the cache and the kernel
// launch interface shared by the host API and the kernels.
//
// Device layout (everything allocated once by okvq_create):
//   unit u = (session * L + layer) * Hkv + kv_head owns P_max = ceil(max_tokens/64)
//   pages of 64 tokens, contiguous: page p of unit u starts at
//   pages + (u * P_max + p) * page_bytes. A page holds, in order,
//     K codes  4 tiles of 16 tokens, each tile 32 lane chunks of 16 B (2-bit) or 32 B (4-bit)
//     V codes  same shape
//     norms    64 fp16, token order
//     stats    64/G groups, each [min 128 fp16 | range 128 fp16] in the stat channel order
//              (TurboQuant keys, G = 0 below: 64 fp16 key norms, token order)
//     tmask    4 bytes, bit m of byte i set when tile i holds a token of modality m,
//              4 bytes of padding, then the 64-bit deletion mask (bit t set: page
//              token t was evicted and is skipped by attention; the same in every
//              (layer, kv head) of a session); the field is 16 B so the page size
//              stays a multiple of 16 B
//   so one decode warp streams one contiguous block per page with a single bulk copy.
//
// Lane chunks: the 32 lanes of a warp running mma.m16n8k16 hold 16x16 / 16x8
// fp16 fragments; lane l owns 32 code pairs j = 0..31 (blk = j/4, r = j%4), each
// pair being the two fp16 halves of one fragment register:
//   K tile (score MMA B operand, channels x tokens; blk = 16-channel block):
//        token = l/4 + 8*(r&1),   channel = 16*blk + 2*(l%4) + 8*(r>>1) + e
//   V tile (value MMA A operand, channels x tokens; blk = 16-channel block):
//        token = 2*(l%4) + 8*(r>>1) + e,   channel = 16*blk + l/4 + 8*(r&1)
// with e = 0/1 the half. Bit position of code e of pair j inside the chunk:
//   4-bit: 8*j + 4*e (pair j = byte j).
//   2-bit V: 4*j + 2*e (pair j = nibble j); a byte holds two pairs and indexes
//        the shared-memory level table.
//   2-bit K: pair j = 8*i + r of word i sits in byte 2*(r/4) + (r&1), nibble
//        (r/2)&1, so the two pairs of one table entry are exactly one score-MMA
//        B fragment (pairs 4kb and 4kb+2, or 4kb+1 and 4kb+3).
//
// Stat channel order: position p = 32*(kb/2) + 8*t + 4*(kb%2) + i (t = 0..3,
// kb = 0..7, i = 0..3) holds channel 16*kb + 2*t + (i&1) + 8*(i>>1): the 8
// channels lane group t needs from a pair of 16-channel blocks are one 16-byte
// chunk, and the four lane groups' chunks are adjacent (one 128-bit shared load
// serves the warp without bank conflicts). Each group stores
// [min 128 fp16 | range 128 fp16].
#pragma once
#include <atomic>
#include <cstddef>
#include <cstdint>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "okvq.h"

namespace okvq {

constexpr int D = 128;
constexpr int PAGE = 64;
constexpr int TILE = 16;
constexpr int MAXM = 3;
constexpr int MAXGQ = 8;

enum : uint32_t { ERR_MODALITY = 1u, ERR_WAIT = 2u };

struct PageLayout {
  int bits, G;
  int lane_bytes;   // 16 or 32
  int tile_bytes;   // 32 * lane_bytes
  int off_v;        // 4 tiles of K codes
  int off_norm;
  int off_stats;
  int off_tmask;    // 4 tile modality masks, then (at +8) the 64-bit deletion mask
  int page_bytes;
};

// G = 0 selects TurboQuant keys: per-token key norms instead of group statistics.
__host__ __device__ inline PageLayout page_layout(int bits, int G) {
  PageLayout L;
  L.bits = bits;
  L.G = G;
  L.lane_bytes = bits * 8;                 // 64 codes * bits / 8
  L.tile_bytes = 32 * L.lane_bytes;
  L.off_v = 4 * L.tile_bytes;
  L.off_norm = 2 * L.off_v;
  L.off_stats = L.off_norm + PAGE * 2;
  L.off_tmask = L.off_stats + (G ? (PAGE / G) * 2 * D * 2 : PAGE * 2);
  L.page_bytes = L.off_tmask + 16;
  return L;
}

// token/channel of code e of pair j in lane l's chunk (see header comment)
__host__ __device__ inline void k_pair_coords(int lane, int j, int e, int &tok, int &ch) {
  int blk = j >> 2, reg = j & 3;
  tok = (lane >> 2) + 8 * (reg & 1);
  ch = 16 * blk + 2 * (lane & 3) + 8 * (reg >> 1) + e;
}
__host__ __device__ inline void v_pair_coords(int lane, int j, int e, int &tok, int &ch) {
  int blk = j >> 2, reg = j & 3;
  tok = 2 * (lane & 3) + 8 * (reg >> 1) + e;
  ch = 16 * blk + (lane >> 2) + 8 * (reg & 1);
}
__host__ __device__ inline int k_code_bit(int bits, int j, int e) {
  if (bits == 4) return 8 * j + 4 * e;
  const int word = j >> 3, r = j & 7;
  return 32 * word + 8 * (2 * (r >> 2) + (r & 1)) + 4 * ((r >> 1) & 1) + 2 * e;
}
__host__ __device__ inline int v_code_bit(int bits, int j, int e) { return bits == 4 ? 8 * j + 4 * e : 4 * j + 2 * e; }

// Inverse of k_code_bit / v_code_bit: the (pair, half) whose code starts at bit b
// of chunk word wi (b a multiple of bits).
__host__ __device__ inline void chunk_code_at(int kind, int bits, int wi, int b, int &j, int &e) {
  if (bits == 4) {
    j = (32 * wi + b) >> 3;
    e = (b >> 2) & 1;
  } else if (kind == 0) {
    const int byte = b >> 3, nib = (b >> 2) & 1;
    e = (b >> 1) & 1;
    j = 8 * wi + 4 * (byte >> 1) + 2 * nib + (byte & 1);
  } else {
    j = (32 * wi + b) >> 2;
    e = (b >> 1) & 1;
  }
}

__host__ __device__ inline int stat_channel(int p) {
  const int k2 = p >> 5, t = (p >> 3) & 3, u = (p >> 2) & 1, i = p & 3;
  return 16 * (2 * k2 + u) + 2 * t + (i & 1) + 8 * (i >> 1);
}
__host__ __device__ inline int stat_pos(int c) {
  const int kb = c >> 4, r = c & 15;
  const int t = (r & 7) >> 1, i = (r & 1) | ((r >> 3) << 1);
  return 32 * (kb >> 1) + 8 * t + 4 * (kb & 1) + i;
}

struct DecodeArgs {
  const __half *q;          // [S][L][Hq][D]
  const uint8_t *pages;
  const __half *tails;      // [2][units][G][D]
  const uint8_t *mod;       // [S][cap]
  const int *segs;          // [nseg][4] = unit, page_begin, page_end, partial slot
  const int *cta_seg;       // [ncta+1]
  const long long *unit_len;// [units] token count
  const int *unit_tail;     // [units] 0/1 current tail buffer
  float *partials;          // [nseg][MAXGQ][2 + MAXM*D]
  int L, Hq, Hkv, M, bits, G;   // G: key group size, 0 = TurboQuant keys
  long long P_max, cap;
  long long units;
  const unsigned char *lut; // [256 code bytes][K 128 B | V 128 B] level table, built by launch_lut
  const float *signs;       // [D] +-1
  uint32_t *err;
};

// The decode kernel's code-byte -> fp16 level table (64 KB), built once per cache.
struct LutArgs {
  unsigned char *out;
  __half klev[16];          // key levels (the value levels for TurboQuant keys)
  __half vlev[16];          // value levels
};

struct CombineArgs {
  const float *partials;
  const int *unit_seg;      // [units+1]
  const uint4 *rot_frag;    // R^T as mma A fragments: [L*Hkv][8 m-tiles][8*M k-steps][32 lanes][hi, lo]
  __half *out;              // [S][L][Hq][D]
  uint32_t *err;
  int L, Hq, Hkv, M;
  long long units;
  const float *far;         // far-memory partials [units][far_split][MAXGQ][FAR_PARTIAL_FLOATS], or null
  int far_split;            // 0: no far memory
};

// Far-memory pseudo tokens (fp16, the original key / value bases) of every unit.
struct FarArgs {
  const __half *q;          // [S][L][Hq][D]
  const __half *k, *v;      // [units][n_far][D]
  const float *mass;        // [units][n_far / per_proto]
  float *partials;          // [units][nsplit][MAXGQ][FAR_PARTIAL_FLOATS]
  uint32_t *err;
  int L, Hq, Hkv;
  int n_far, per_proto;
  int nsplit, chunk;        // splits per unit, tokens per split
  long long units;
};

constexpr int PARTIAL_FLOATS = 2 + MAXM * D;   // m, l, o[M][D]
constexpr int FAR_PARTIAL_FLOATS = 2 + D;       // m, l, o[D] (original value basis)
constexpr int DEAD_OFF = 8;                     // deletion mask: page offset off_tmask + DEAD_OFF

// Compaction granule: the tokens that move together (a key group, whose statistics
// serve all its members, or one 16-token tile for TurboQuant keys).
__host__ __device__ inline int compaction_granule(int KG) { return KG ? KG : TILE; }

// Bytes of one granule of one (layer, kv head) in the gather scratch: K code tiles,
// V code tiles, value norms, key statistics (one group) or key norms, tile masks;
// rounded up to 16 B.
__host__ __device__ inline int granule_payload(const PageLayout &PL, int KG) {
  const int gran = compaction_granule(KG), nt = gran / TILE;
  const int b = 2 * nt * PL.tile_bytes + 2 * gran + (KG ? 2 * D * 2 : 2 * gran) + nt;
  return (b + 15) & ~15;
}

struct MoveArgs {
  uint8_t *pages;
  uint8_t *mod;             // [S][cap]
  const int *moves;         // [n][2] (source granule, destination granule), this batch
  uint8_t *scratch;         // [n][LH + 1][stride]: per unit payloads, then the modality ids
  int n, LH, KG, session;
  int stride;               // bytes per (move, unit) slot, >= granule_payload and the granule's ids
  int scatter;              // 0: pages -> scratch, 1: scratch -> pages
  long long P_max, cap;
  PageLayout PL;
};

struct PageMetaArgs {
  uint8_t *pages;
  const unsigned long long *dead;   // [P_max] this session's deletion masks
  int LH, session;
  long long p0;             // first page rewritten
  long long T;              // session length: tile masks of tiles at or past it are cleared
  long long P_max;
  PageLayout PL;
};

// True for device or managed memory (a host query, no caching).
inline bool is_device_memory(const void *p) {
  if (!p) return false;
  cudaPointerAttributes at{};
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    (void)cudaGetLastError();
    return false;
  }
  return at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged;
}

// Kernel attributes belong to a device: run `set` once per device ordinal (the
// current device; ordinals >= 64 run it on every call). `done` holds one bit per
// device.
template <class Fn>
cudaError_t once_per_device(std::atomic<uint64_t> &done, Fn set) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = dev >= 0 && dev < 64 ? (1ull << dev) : 0ull;
  if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
  e = set();
  if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_acq_rel);
  return e;
}

cudaError_t launch_decode(const DecodeArgs &a, int n_cta, cudaStream_t s);
cudaError_t launch_combine(const CombineArgs &a, cudaStream_t s);
cudaError_t launch_lut(int bits, const LutArgs &a, cudaStream_t s);
constexpr size_t LEVEL_TABLE_BYTES = 256 * 256;
size_t decode_smem_bytes(int bits, int G);
int decode_warps(int bits);   // warps per decode CTA: a CTA takes its pages in turns of this many
cudaError_t launch_move(const MoveArgs &a, cudaStream_t s);
cudaError_t launch_far(const FarArgs &a, cudaStream_t s);
int far_pass_tokens();        // pseudo tokens one pass of the far kernel's warps takes
cudaError_t launch_page_meta(const PageMetaArgs &a, int n_pages, cudaStream_t s);

}  // namespace okvq
