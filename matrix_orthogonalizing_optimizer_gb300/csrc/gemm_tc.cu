// Batched 16-bit (bf16 or fp16) GEMM on the 5th-generation tensor cores (tcgen05 + TMEM +
// TMA), sm_103a. A and B share one type (kind::f16 takes both bf16 or both fp16); the addend C
// and the outputs D, D2 may each be bf16 or fp16.
//
// A cluster of two CTAs (a CTA pair on neighbouring SMs) computes one 256 x 256 output
// tile with 2-CTA MMAs (tcgen05.mma.cta_group::2, M = 256, N = 256, K = 16): each CTA
// stages its 128 rows of A and its 128 columns of B, and holds its 128 x 256 half of the
// fp32 accumulator in its own tensor memory (Dion3 appendix C.1: 256 x 256 cluster tiles,
// 2-CTA collaboration, two accumulators so the epilogue overlaps the next main loop).
// Persistent pairs walk a list of tiles: every tile of a rectangular product, or the
// upper-triangle tiles of a symmetric one (Dion3 sec. 5, "Triangular Scheduler").
//
// Warp roles in each CTA:
//   warp 0    TMA producer: 64-wide K slices into a ring of stages (128-byte swizzle; a
//             K-major operand is one 128 x 64 box, an MN-major one two 64 x 64 boxes);
//             completion is signalled on the leader CTA's stage barrier. Warp 0 loads the
//             even K slices of the pair's sequence, warp 11 (a second producer) the odd ones.
//   warp 1    TMEM allocation (both CTAs) and, in the leader CTA, the MMA issuer.
//   warp 2    C-tile loader: TMA loads of the addend C, chunk by chunk, into a small ring
//             as soon as the epilogue frees each buffer.
//   warps 3-10 epilogue, two warps per TMEM lane quarter (thread = row, each warp 32 of a
//             chunk's 64 columns): tcgen05.ld of the accumulator, alpha/beta with the C tile,
//             result staged in 128-byte-swizzled shared memory and written with TMA stores
//             in 64-column chunks; off-diagonal tiles of symmetric products are also stored
//             transposed at the mirrored position (through the same staging buffer),
//             diagonal tiles once (Dion3 sec. 5 "Writing to the Transposed Tile",
//             appendix C.1).
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdio>
#include <cstdlib>
#include <mutex>
#include <vector>

#include "common.cuh"
#include "gemm.h"

namespace gns {

namespace tc {

constexpr int TM = 128;                          // accumulator rows per CTA
constexpr int BN = 128;                          // B columns staged per CTA
constexpr int TK = 64;                           // K slice per stage
#ifndef GNS_TC_OUTBUFS
#define GNS_TC_OUTBUFS 2
#endif
// staging buffers for output (and mirror) chunks: with two, a chunk's stores drain while the
// next chunk is staged
constexpr int OUT_BUFS = GNS_TC_OUTBUFS;
constexpr int A_BYTES = TM * TK * 2;             // 16 KiB
constexpr int STAGE_BYTES = (TM + BN) * TK * 2;  // 32 KiB per CTA
constexpr int CHUNK = 64;                        // epilogue columns per chunk
constexpr int BOX_BYTES = 64 * 64 * 2;           // one 64 x 64 16-bit box, 128-byte swizzle
constexpr int CHUNK_BYTES = 2 * BOX_BYTES;       // 128 x 64 (or 64 x 128) elements
constexpr int C_WARP = 2;                        // loads the C tile ahead of the epilogue
constexpr int FIRST_EPI_WARP = 3;
constexpr int EPI_WARPS = 8;                     // two per TMEM lane quarter
constexpr int EPI_THREADS = 32 * EPI_WARPS;
// A second TMA producer in a warp of its own takes the odd K slices: two issuing threads
// keep more operand loads in flight than one (warps 0 and PROD2_WARP; a producer sharing a
// warp with another role would run divergent with it).
constexpr int PROD2_WARP = FIRST_EPI_WARP + EPI_WARPS;
constexpr int NUM_THREADS = 32 * (FIRST_EPI_WARP + EPI_WARPS + 1);
constexpr int MAX_PROB = 24;                     // stages of one launch

// Tile geometry of a CTA group: CG = 2 (a CTA pair, 2-CTA MMAs, 256 x 256 tiles) or CG = 1
// (one CTA, 128 x 128 tiles, for products of at most 128 rows: a 256 x 256 tile would
// compute 4x the useful work of an n <= 128 Gram product). Per CTA the operand staging is the
// same (128 rows of A, 128 columns of B per 64-wide K slice); the accumulator is TILE
// columns wide, two of them in tensor memory.
template <int CG>
struct Geo {
  static constexpr int TILE = 128 * CG;             // tile rows = tile columns
  static constexpr int NCH = TILE / CHUNK;          // epilogue chunks per tile
  static constexpr int TMEM_COLS = 2 * TILE;        // two fp32 accumulators
  static constexpr int KSH = CG == 2 ? 2 : 1;       // log2 of 64-wide K slices per tile edge
};
constexpr int BAR_BYTES = 2048;
// In the barrier area: for row-mapped outputs, two buffers (by tile parity) of the W row of
// each tile row, the next tile's written during the current one; then a ring of the
// epilogue's per-tile parameters (TileInfo), filled ahead by one lane of the C-loader warp, and
// its barriers: full (the entry is written), stored (the epilogue's stores of the tile have
// landed) and empty (the epilogue and the publishing lane are done with the entry).
constexpr int RM_IDX_OFF = 256;
constexpr int INFO_RING = 8;
constexpr int INFO_OFF = RM_IDX_OFF + 2 * TM * 4;
constexpr int INFO_BAR_OFF = INFO_OFF + INFO_RING * 48;
static_assert(INFO_BAR_OFF + 3 * INFO_RING * 8 <= BAR_BYTES, "tile-info ring");

// Shared-memory plan of a kernel with STAGES operand stages and a ring of C_BUFS C chunks.
// Two plans are compiled: a deeper operand ring (5 stages, 2 C chunks) for launches of short
// tiles (few K slices per tile: the ring also covers the switch to the next tile, and the
// second C chunk keeps the addend of the n x n products loading a chunk ahead of their
// epilogues, which otherwise hold the accumulator the next tile waits for; 6 stages with one
// C chunk measured 2 % slower on the 24 x 1024 x 4096 step); a shallow one (4 stages, 4 C
// chunks) on launches of long tiles, where a deeper ring only keeps more operand lines in
// flight and costs L2 reuse.
template <int STAGES_, int C_BUFS_>
struct Plan {
  static constexpr int STAGES = STAGES_;
  static constexpr int C_BUFS = C_BUFS_;
  static constexpr int OFF_SC = STAGES * STAGE_BYTES;  // C chunks (ring of C_BUFS)
  static constexpr int OFF_SD = OFF_SC + C_BUFS * CHUNK_BYTES;
  static constexpr int OFF_BAR = OFF_SD + OUT_BUFS * CHUNK_BYTES;
  static constexpr int SMEM_BYTES = 1024 + OFF_BAR + BAR_BYTES;
  static_assert(SMEM_BYTES <= 232448, "shared memory budget");
  static_assert((2 * STAGES + 4 + 2 * C_BUFS) * 8 + 16 <= RM_IDX_OFF, "barrier area");
};
using DeepPlan = Plan<5, 2>;
using ShallowPlan = Plan<4, 4>;
// Launches whose tiles average at most DEEP_MAX_SLICES_PER_TILE K slices take the deep plan,
// and so do those of at most DEEP_SMALL_BATCH matrices per product whose tiles average at most
// DEEP_MAX_SLICES_SMALL_BATCH (measured: 32 x 4096^2 standard NS 7 % and 32 x 11008 x 4096
// Gram NS 8 % faster on the deep plan; 64-matrix and larger batches of the same shapes, and
// the 256 x 2048 x 8192 MoE batch, 3-20 % slower).
constexpr int DEEP_MAX_SLICES_PER_TILE = 24;
constexpr int DEEP_SMALL_BATCH = 32;
constexpr int DEEP_MAX_SLICES_SMALL_BATCH = 96;

// Partial sums per matrix a problem's norm scale is formed from (scale_part).
constexpr int SCALE_NPART = 32;

struct Problem {
  CUtensorMap tmA;
  CUtensorMap tmB;
  CUtensorMap tmA2;  // the other major-ness of A / B (upper-stored symmetric operands)
  CUtensorMap tmB2;
  CUtensorMap tmC;
  CUtensorMap tmD;
  CUtensorMap tmD2;
  int a_mn, b_mn;
  int kblocks;
  int tiles_m, tiles_n, sym;
  int tiles_per_mat;
  float alpha, beta, gamma;
  int alpha_pow, beta_pow;
  const float* scale;
  int has_c, c_trans, d_trans, has_d2;
  int diag_limit;
  int check_finite;
  int a_upper, b_upper, mirror_out;
  int ab_f16, c_f16, d_f16;  // 16-bit element types: fp16 (1) or bf16 (0)
  int c_mode, d_mode;        // chunk modes of the C loads and of the direct D / D2 stores
  uint32_t dep_mask;  // earlier problems whose tiles of the same matrix must be complete
  int ctr_off;        // this problem's completion counters: counters[ctr_off + b]
  int publish;        // a later problem of the launch depends on this one: publish completions
  int scale_part;     // scale holds SCALE_NPART partial sums per matrix (16-byte aligned), not scales
};
// (the parameter block holds up to MAX_PROB of these: the fields fit in the 1024 bytes that
// the seven 64-byte-aligned tensor maps round the struct up to)
static_assert(sizeof(Problem) == 1024, "Problem size");

// The launch's tiles form a sequence of segments, each the tiles of problem p for the
// matrices b0 .. b0 + nb - 1 (matrix-major, then tile): seg_pb = p << 24 | b0, seg_tile =
// index of its first tile (nb follows from the next segment's start). The host orders the
// segments so that every tile depends only on tiles earlier in the sequence.
constexpr int MAX_SEG = 576;

// A problem whose output rows go through a row map (the fractional update's
// W[S] <- beta W[S] + alpha O): the epilogue threads read C and write D (the same matrix) with
// plain 16-byte global accesses, row i of the product at row map[b * map_stride + i] of
// matrix b, instead of TMA tiles. rows: valid product rows; cols: columns of D.
struct RowMapOut {
  int prob;  // -1: none
  int map_stride;
  const int32_t* map;
  void* ptr;
  long long ld, stride;
  int rows, cols;
  int has_c;
};

struct Params {
  Problem prob[MAX_PROB];
  RowMapOut rmo;
  float scale_eps;  // the eps of every scale formed from partial sums in the launch
  int nprob;
  int total_tiles;
  int nseg;
  int* status;
  int* counters;  // per (problem, matrix): CTA-halves of tiles completed (zero at launch)
  uint32_t seg_pb[MAX_SEG];
  int seg_tile[MAX_SEG];
};

// Bounded wait until every problem this tile depends on has finished matrix b.
template <int CG>
__device__ __forceinline__ bool wait_deps(const Params& P, const Problem& pr, int b, volatile int* abort_flag) {
  uint32_t m = pr.dep_mask;
  while (m) {
    const int d = __ffs(m) - 1;
    m &= m - 1;
    const Problem& pd = P.prob[d];
    if (!wait_counter(P.counters + pd.ctr_off + b, CG * pd.tiles_per_mat, abort_flag, P.status)) return false;
  }
  return true;
}

// Bounded wait until the scout lane has found this tile's dependencies complete (its
// published index reaches `tile`); then order later TMA reads after that observation.
__device__ __forceinline__ bool wait_ready(volatile int* ready, int tile, volatile int* abort_flag, int* status) {
  if (*ready < tile) {
    const uint64_t t0 = global_timer_ns();
    for (uint32_t i = 1;; ++i) {
      if (*ready >= tile) break;
      if ((i & 63u) == 0u) {
        if (*abort_flag) return false;
        if (global_timer_ns() - t0 > GNS_WAIT_TIMEOUT_NS) {
          *abort_flag = 1;
          set_status(status, GNS_DEVST_TIMEOUT);
          return false;
        }
      }
    }
  }
  __threadfence_block();
  fence_proxy_async_global();
  return true;
}

// Major-ness of the A (B) slice of 64-wide K block kb for tile row I (column J). An operand
// that is the upper triangle of a symmetric matrix (tile blocks at or above the diagonal) is
// read from the mirrored block, with the other major-ness, wherever the block it would read
// lies below the diagonal.
// The per-product fields a K loop reads, copied into registers once per tile: the loops'
// inline assembly clobbers memory, which would otherwise reload them at every K slice.
struct KLoop {
  int kblocks, a_mn, b_mn, a_upper, b_upper, ab_f16, ksh;
};
__device__ __forceinline__ int a_major(const KLoop& pr, int I, int kb) {
  const int kbl = kb >> pr.ksh;
  const bool lower = pr.a_mn ? (kbl > I) : (I > kbl);
  return pr.a_mn ^ ((pr.a_upper && lower) ? 1 : 0);
}
__device__ __forceinline__ int b_major(const KLoop& pr, int J, int kb) {
  const int kbl = kb >> pr.ksh;
  const bool lower = pr.b_mn ? (kbl > J) : (J > kbl);
  return pr.b_mn ^ ((pr.b_upper && lower) ? 1 : 0);
}

struct TileCoord {
  int p, b, I, J;
};

// What the roles need of one tile, decoded and scaled ahead of them: decoding reads the
// parameter block with tile-dependent indices, and the per-matrix scale is a global load, so
// done at the top of each tile they kept the epilogue and the MMA issuer waiting between
// tiles (the launch's bottleneck on tiles of few K slices).
enum : uint32_t {
  TI_HAS_C = 1u << 8, TI_MIRROR = 1u << 9, TI_DIAG = 1u << 10, TI_C_TRANS = 1u << 11, TI_C_F16 = 1u << 12,
  TI_D_TRANS = 1u << 13, TI_D_F16 = 1u << 14, TI_CHECK = 1u << 15, TI_HAS_D2 = 1u << 16, TI_PUBLISH = 1u << 17,
  TI_ROWMAP = 1u << 18, TI_DMODE_SHIFT = 19  // bits 0-7: the problem; 19-20: the D chunk mode
};
enum : uint32_t { KF_A_MN = 1u, KF_B_MN = 2u, KF_A_UPPER = 4u, KF_B_UPPER = 8u, KF_AB_F16 = 16u, KF_DEP = 32u,
                  KF_CMODE_SHIFT = 6 };
struct TileInfo {
  uint32_t pf;     // problem and flags
  int b;           // matrix
  uint32_t ij;     // tile row I (low half) and column J (high half)
  int ctr_off;     // the problem's completion counters
  float alpha, beta, gamma;
  int diag_limit;
  int kblocks;     // K slices
  uint32_t kf;     // operand major-ness and types, dependencies, C chunk mode
  int pad[2];
};
static_assert(sizeof(TileInfo) == 48, "tile-info entry");

// s0: a segment index at or below the tile's (every role walks its tiles in increasing
// order, so the previous tile's segment is a valid start); *seg receives the tile's.
__device__ __forceinline__ TileCoord decode_tile(const Params& P, int tile, int* seg) {
  TileCoord tc;
  int s = *seg;
  while (s + 1 < P.nseg && tile >= P.seg_tile[s + 1]) ++s;
  *seg = s;
  const uint32_t pb = P.seg_pb[s];
  const int p = (int)(pb >> 24);
  const Problem& pr = P.prob[p];
  int t = tile - P.seg_tile[s];
  tc.p = p;
  const int bi = t / pr.tiles_per_mat;
  tc.b = (int)(pb & 0xFFFFFFu) + bi;
  t -= bi * pr.tiles_per_mat;
  if (pr.sym) {
    int i = 0;
    while (t >= pr.tiles_m - i) {
      t -= pr.tiles_m - i;
      ++i;
    }
    tc.I = i;
    tc.J = i + t;
  } else {
    tc.I = t / pr.tiles_n;
    tc.J = t - tc.I * pr.tiles_n;
  }
  return tc;
}

// A tile's coordinates and K loop from its TileInfo entry (copied out of shared memory once).
struct TileHead {
  TileCoord c;
  KLoop kl;
  uint32_t pf, kf;
};
__device__ __forceinline__ TileHead tile_head(const TileInfo* e, int ksh) {
  TileHead h;
  h.pf = e->pf;
  h.kf = e->kf;
  const uint32_t ij = e->ij;
  h.c.p = (int)(h.pf & 0xFFu);
  h.c.b = e->b;
  h.c.I = (int)(ij & 0xFFFFu);
  h.c.J = (int)(ij >> 16);
  h.kl.ksh = ksh;
  h.kl.kblocks = e->kblocks;
  h.kl.a_mn = (h.kf & KF_A_MN) != 0;
  h.kl.b_mn = (h.kf & KF_B_MN) != 0;
  h.kl.a_upper = (h.kf & KF_A_UPPER) != 0;
  h.kl.b_upper = (h.kf & KF_B_UPPER) != 0;
  h.kl.ab_f16 = (h.kf & KF_AB_F16) != 0;
  return h;
}

__device__ __forceinline__ float powi(float s, int p) { return p == 0 ? 1.f : (p == 1 ? s : s * s); }

// Byte offset of element (tile row r in [0,128), chunk column c in [0,64)) in a staged chunk:
// "direct" keeps the tile's orientation (two 64-row boxes), "transposed" stores the chunk as
// its transpose (64 rows x 128 columns, two 64-column boxes). Both follow the 128-byte
// swizzle of the TMA boxes: 16-byte unit u of box row y lives at unit u ^ (y & 7).
__device__ __forceinline__ uint32_t off_direct(int r, int c) {
  const int y = r & 63;
  return (uint32_t)((r >> 6) * BOX_BYTES + y * 128 + (((c >> 3) ^ (y & 7)) << 4) + ((c & 7) << 1));
}
__device__ __forceinline__ uint32_t off_trans(int r, int c) {
  const int x = r & 63;
  return (uint32_t)((r >> 6) * BOX_BYTES + c * 128 + (((x >> 3) ^ (c & 7)) << 4) + ((x & 7) << 1));
}

// One chunk = rows [row0, row0+128) x cols [col0, col0+64) of the matrix (mode 0: two
// 64 x 64 boxes; mode 2: one 128-row box, same shared-memory layout, for maps encoded with
// 128-row boxes), or rows [col0, col0+64) x cols [row0, row0+128) (mode 1, transposed: two
// 64 x 64 boxes). Every TMA box costs the SM's TMA unit a roughly fixed time, so chunks
// take one box wherever the map allows.
__device__ __forceinline__ void chunk_load(uint8_t* s, const CUtensorMap* map, uint64_t* bar, int mode, int row0,
                                           int col0, int b) {
  if (mode == 2) {
    tma_load_3d(s, map, bar, col0, row0, b);
  } else if (mode == 0) {
    tma_load_3d(s, map, bar, col0, row0, b);
    tma_load_3d(s + BOX_BYTES, map, bar, col0, row0 + 64, b);
  } else {
    tma_load_3d(s, map, bar, row0, col0, b);
    tma_load_3d(s + BOX_BYTES, map, bar, row0 + 64, col0, b);
  }
}
__device__ __forceinline__ void chunk_store(const uint8_t* s, const CUtensorMap* map, int mode, int row0, int col0,
                                            int b) {
  if (mode == 2) {
    tma_store_3d(map, s, col0, row0, b);
  } else if (mode == 0) {
    tma_store_3d(map, s, col0, row0, b);
    tma_store_3d(map, s + BOX_BYTES, col0, row0 + 64, b);
  } else {
    tma_store_3d(map, s, row0, col0, b);
    tma_store_3d(map, s + BOX_BYTES, row0 + 64, col0, b);
  }
}

// The epilogue's arithmetic runs on value pairs (the paired fp32 instructions, each element
// rounded as its scalar form would be): its warps share the SMs' issue slots with the
// single-thread producer and MMA roles, so every instruction saved there is main-loop time.
//
// o += beta * C for 32 values held two per word (fp16 when f16, else bf16); the element type
// is decided once per chunk, not per value.
__device__ __forceinline__ void axpy_h16x2(float2 (&o)[16], const uint32_t (&cw)[16], float beta, int f16) {
  const float2 b2 = make_float2(beta, beta);
  if (f16) {
#pragma unroll
    for (int i = 0; i < 16; ++i) o[i] = __ffma2_rn(b2, __half22float2(*reinterpret_cast<const __half2*>(&cw[i])), o[i]);
  } else {
#pragma unroll
    for (int i = 0; i < 16; ++i)  // bf16 -> fp32 is exact: the bits move up 16 places
      o[i] = __ffma2_rn(b2, make_float2(__uint_as_float(cw[i] << 16), __uint_as_float(cw[i] & 0xFFFF0000u)), o[i]);
  }
}

// 32 fp32 values rounded to nearest even, two per word (the first in the low half), with
// the paired conversion instructions.
__device__ __forceinline__ void pack_h16x2(const float2 (&o)[16], uint32_t (&pk)[16], int f16) {
  if (f16) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const __half2 h = __float22half2_rn(o[i]);
      pk[i] = *reinterpret_cast<const uint32_t*>(&h);
    }
  } else {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const __nv_bfloat162 h = __float22bfloat162_rn(o[i]);
      pk[i] = *reinterpret_cast<const uint32_t*>(&h);
    }
  }
}

// One operand box of a K slice into this CTA's stage; completion is signalled on the stage
// barrier at shared::cluster address bar (the pair leader's for CG = 2, with .cta_group::2).
template <int CG>
__device__ __forceinline__ void op_load(void* dst, const CUtensorMap* map, uint32_t bar, int c0, int c1, int c2) {
  if constexpr (CG == 2) {
    tma_load_3d_pair(dst, map, bar, c0, c1, c2);
  } else {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
        : "memory");
  }
}

// Releases an accumulator to the group's MMA issuer: a remote arrival on the leader's barrier
// for a CTA pair, a local one for a single CTA.
template <int CG>
__device__ __forceinline__ void acc_release(uint32_t bar) {
  if constexpr (CG == 2)
    mbar_arrive_cluster(bar);
  else
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// The addend of one epilogue thread's row segment of a row-mapped chunk: W row wr (-1: none),
// columns col .. col + 31, as four 16-byte vectors (zeros past the matrix's columns). Loaded
// straight into the registers the epilogue adds it from, a chunk ahead: a warp reads 32 rows'
// 64-byte segments, whole 32-byte sectors.
__device__ __forceinline__ void rowmap_own_load(uint4 (&cv)[4], const uint16_t* base, long long ld, int wr, int col,
                                                int cols) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int c = col + 8 * q;
    uint4 w = make_uint4(0u, 0u, 0u, 0u);
    if (wr >= 0 && c < cols) {
      const uint16_t* p = base + (long long)wr * ld + c;
      if (c + 8 <= cols) {
        w = *reinterpret_cast<const uint4*>(p);
      } else {
        uint32_t e[4] = {0u, 0u, 0u, 0u};
        for (int j = 0; j < 8 && c + j < cols; ++j) e[j >> 1] |= (uint32_t)p[j] << (16 * (j & 1));
        w = make_uint4(e[0], e[1], e[2], e[3]);
      }
    }
    cv[q] = w;
  }
}

// Row-mapped chunks: 128 rows x 64 columns of W whose rows are rm_idx[0..127] (-1: none).
// Thread t of the 256 epilogue threads stores the 16-byte vectors v = t + 256 i (i < 4): row
// v / 8, columns 8 (v % 8) .. +7 of the chunk, so a warp covers four whole 128-byte row
// segments per access. Vectors past the matrix's columns are partial (not written).
__device__ __forceinline__ void rowmap_chunk_store(const uint8_t* sd, void* ptr, long long boff, long long ld,
                                                   const int* rm_idx, int t, int col0, int cols) {
  uint16_t* const base = static_cast<uint16_t*>(ptr) + boff;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int v = t + 256 * i;
    const int row = v >> 3;
    const int col = col0 + (v & 7) * 8;
    const int wr = rm_idx[row];
    if (wr < 0 || col >= cols) continue;
    const uint4 w = *reinterpret_cast<const uint4*>(sd + off_direct(row, (v & 7) * 8));
    uint16_t* q = base + (long long)wr * ld + col;
    if (col + 8 <= cols) {
      *reinterpret_cast<uint4*>(q) = w;
    } else {
      const uint32_t e[4] = {w.x, w.y, w.z, w.w};
      for (int j = 0; j < 8 && col + j < cols; ++j) q[j] = (uint16_t)(e[j >> 1] >> (16 * (j & 1)));
    }
  }
}

// PS: the launch forms scales from partial sums (scale_part) and is a programmatic dependent
// launch. Launches without either run an instance without that code: on launches of many short
// tiles, where the tile-info lane is on the critical path, it measured a few per cent slower.
template <class L, int CG, bool PS>
__global__ void __launch_bounds__(NUM_THREADS, 1) gemm_kernel(const __grid_constant__ Params P) {
  constexpr int TT = Geo<CG>::TILE;
  constexpr int NCHUNK = Geo<CG>::NCH;
  constexpr int TMEM_COLS = Geo<CG>::TMEM_COLS;
  constexpr int STAGES = L::STAGES;
  constexpr int C_BUFS = L::C_BUFS;
  constexpr int OFF_SC = L::OFF_SC;
  constexpr int OFF_SD = L::OFF_SD;
  constexpr int OFF_BAR = L::OFF_BAR;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* stages = smem;
  uint8_t* SC = smem + OFF_SC;
  uint8_t* SD = smem + OFF_SD;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
  uint64_t* full = bars;
  uint64_t* empty = bars + STAGES;
  uint64_t* tfull = bars + 2 * STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* cfull = tempty + 2;
  uint64_t* cempty = cfull + C_BUFS;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(cempty + C_BUFS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* epi_flag = abort_flag + 1;
  volatile int* ready_tile = abort_flag + 2;  // highest tile of this pair whose inputs are complete
  TileInfo* const info = reinterpret_cast<TileInfo*>(smem + OFF_BAR + INFO_OFF);
  uint64_t* const info_full = reinterpret_cast<uint64_t*>(smem + OFF_BAR + INFO_BAR_OFF);
  uint64_t* const info_empty = info_full + INFO_RING;
  uint64_t* const info_stored = info_empty + INFO_RING;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // a "pair" is the CTA group of one tile: two CTAs of a cluster, or one CTA
  const uint32_t rank = CG == 2 ? cluster_ctarank() : 0u;
  const int pair = blockIdx.x / CG;
  const int npairs = gridDim.x / CG;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], CG * EPI_WARPS);  // one arrival per epilogue warp of the group
    }
    for (int q = 0; q < C_BUFS; ++q) {
      mbar_init(&cfull[q], 1);
      mbar_init(&cempty[q], EPI_WARPS);
    }
    for (int q = 0; q < INFO_RING; ++q) {
      mbar_init(&info_full[q], 1);
      mbar_init(&info_empty[q], 2);
      mbar_init(&info_stored[q], 1);
    }
    *abort_flag = 0;
    *epi_flag = 1;
    *ready_tile = -1;
    mbar_fence_init();
  }
  if (warp == 0 && lane == 0) {
    for (int p = 0; p < P.nprob; ++p) {
      tma_prefetch_desc(&P.prob[p].tmA);
      tma_prefetch_desc(&P.prob[p].tmB);
    }
  }
  if (warp == 1) {
    if constexpr (CG == 2) {
      tmem_alloc2(tmem_slot, TMEM_COLS);
      tmem_relinquish2();
    } else {
      tmem_alloc(tmem_slot, TMEM_COLS);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  __syncthreads();
  if constexpr (CG == 2) cluster_sync_all();  // the peer's barriers are initialised before any remote arrival
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // everything above touches only this CTA pair's shared memory and TMEM: with a programmatic
  // launch it overlaps the end of the kernel ahead, whose results are read from here on
  if constexpr (PS) grid_dep_wait();

  if (warp == 0 || warp == PROD2_WARP) {
    if (lane == 0) {
      // ---------------- TMA producers (both CTAs): even K slices / odd K slices ----------------
      const int pid = warp == 0 ? 0 : 1;
      int* const status = P.status;
      // stage barriers: the leader's for a CTA pair
      const uint32_t full0 = CG == 2 ? mapa_shared(smem_u32(&full[0]), 0) : smem_u32(&full[0]);
      uint32_t g = 0;  // K slices of this pair so far: producer g & 1 takes slice g
      int s = 0;
      uint32_t ph = 0;
      bool ok = true;
      int local = 0;
      for (int tile = pair; ok && tile < P.total_tiles; tile += npairs, ++local) {
        const int islot = local % INFO_RING;
        if (!mbar_wait(&info_full[islot], (local / INFO_RING) & 1u, abort_flag, status)) break;
        const TileHead h = tile_head(&info[islot], Geo<CG>::KSH);
        const TileCoord c = h.c;
        const KLoop kl = h.kl;
        const Problem& pr = P.prob[c.p];  // (tensor-map addresses only)
        const int m0 = c.I * TT + (int)rank * TM;
        const int n0 = c.J * TT + (int)rank * BN;
        const CUtensorMap* const tmA = &pr.tmA;
        const CUtensorMap* const tmA2 = &pr.tmA2;
        const CUtensorMap* const tmB = &pr.tmB;
        const CUtensorMap* const tmB2 = &pr.tmB2;
        if ((h.kf & KF_DEP) && !wait_ready(ready_tile, tile, abort_flag, status)) break;
        for (int kb = 0; kb < kl.kblocks; ++kb) {
          if ((g++ & 1u) != (uint32_t)pid) {  // the other producer's slice
            if (++s == STAGES) {
              s = 0;
              ph ^= 1u;
            }
            continue;
          }
          if (!mbar_wait(&empty[s], ph ^ 1u, abort_flag, status)) {
            ok = false;
            break;
          }
          if (rank == 0) mbar_arrive_expect_tx(&full[s], CG * STAGE_BYTES);
          const uint32_t fb = full0 + 8u * (uint32_t)s;
          uint8_t* sa = stages + s * STAGE_BYTES;
          uint8_t* sb = sa + A_BYTES;
          const int k0 = kb * TK;
          const int amn = a_major(kl, c.I, kb), bmn = b_major(kl, c.J, kb);
          const CUtensorMap* ma = amn == kl.a_mn ? tmA : tmA2;
          const CUtensorMap* mb = bmn == kl.b_mn ? tmB : tmB2;
          if (!amn) {
            op_load<CG>(sa, ma, fb, k0, m0, c.b);
          } else {
            op_load<CG>(sa, ma, fb, m0, k0, c.b);
            op_load<CG>(sa + BOX_BYTES, ma, fb, m0 + 64, k0, c.b);
          }
          if (!bmn) {
            op_load<CG>(sb, mb, fb, k0, n0, c.b);
          } else {
            op_load<CG>(sb, mb, fb, n0, k0, c.b);
            op_load<CG>(sb + BOX_BYTES, mb, fb, n0 + 64, k0, c.b);
          }
          if (++s == STAGES) {
            s = 0;
            ph ^= 1u;
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      // ---------------- MMA issuer (leader CTA) ----------------
      int* const status = P.status;
      const uint32_t stages_u = smem_u32(stages);
      int s = 0;
      uint32_t ph = 0;
      bool ok = true;
      int local = 0;
      for (int tile = pair; ok && tile < P.total_tiles; tile += npairs, ++local) {
        const int islot = local % INFO_RING;
        if (!mbar_wait(&info_full[islot], (local / INFO_RING) & 1u, abort_flag, status)) break;
        const TileHead h = tile_head(&info[islot], Geo<CG>::KSH);
        const TileCoord c = h.c;
        const KLoop kl = h.kl;
        const int acc = local & 1;
        const uint32_t aph = (local >> 1) & 1;
        if (!mbar_wait(&tempty[acc], aph ^ 1u, abort_flag, status)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * TT;
        for (int kb = 0; kb < kl.kblocks; ++kb) {
          const int amn = a_major(kl, c.I, kb), bmn = b_major(kl, c.J, kb);
          const uint32_t idesc = idesc_f16kind_f32(TT, TT, amn, bmn, kl.ab_f16);
          if (!mbar_wait(&full[s], ph, abort_flag, status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = stages_u + (uint32_t)s * STAGE_BYTES;
          const uint32_t sb = sa + A_BYTES;
          // descriptors of the slice's first K=16 step; the next steps advance the start
          // address field (16-byte units): 32 bytes along K for a K-major operand, 16 rows of
          // 128 bytes for an MN-major one (stage addresses stay far below the field's 256 KiB)
          const uint64_t ad0 = amn ? sdesc_sw128(sa, BOX_BYTES, 1024) : sdesc_sw128(sa, 16, 1024);
          const uint64_t bd0 = bmn ? sdesc_sw128(sb, BOX_BYTES, 1024) : sdesc_sw128(sb, 16, 1024);
          const uint64_t astep = amn ? 2048 / 16 : 32 / 16;
          const uint64_t bstep = bmn ? 2048 / 16 : 32 / 16;
#pragma unroll
          for (int kk = 0; kk < TK / 16; ++kk) {
            if constexpr (CG == 2)
              umma2_f16kind(d_tmem, ad0 + astep * kk, bd0 + bstep * kk, idesc, (kb | kk) != 0 ? 1u : 0u);
            else
              umma_f16kind(d_tmem, ad0 + astep * kk, bd0 + bstep * kk, idesc, (kb | kk) != 0 ? 1u : 0u);
          }
          if constexpr (CG == 2)
            umma2_commit_multicast(&empty[s], 0x3);
          else
            umma_commit(&empty[s]);
          if (++s == STAGES) {
            s = 0;
            ph ^= 1u;
          }
        }
        if (ok) {
          if constexpr (CG == 2)
            umma2_commit_multicast(&tfull[acc], 0x3);
          else
            umma_commit(&tfull[acc]);
        }
      }
    }
  } else if (warp == C_WARP) {
    if (lane == 1) {
      // ---------------- dependency scout (both CTAs) ----------------
      // Walks this pair's tiles ahead of the producer and the C loader, waits (bounded) on
      // the completion counters of the problems each tile depends on, and publishes the
      // highest tile whose inputs are complete, so the L2 round trips of those checks stay
      // off the producer's path.
      int seg = 0;
      for (int tile = pair; tile < P.total_tiles; tile += npairs) {
        const TileCoord c = decode_tile(P, tile, &seg);
        const Problem& pr = P.prob[c.p];
        if (pr.dep_mask && !wait_deps<CG>(P, pr, c.b, abort_flag)) break;
        __threadfence_block();
        *ready_tile = tile;
      }
    }
    if (lane == 2) {
      // ---------------- tile-info lane (both CTAs) ----------------
      // Decodes this pair's tiles and the epilogue's per-tile parameters into the TileInfo
      // ring, up to INFO_RING tiles ahead of the epilogue.
      int seg = 0, local = 0;
      const float* sc_part = nullptr;  // the last scale formed from partial sums, and its matrix
      int sc_b = -1;
      float sc_last = 0.f;
      for (int tile = pair; tile < P.total_tiles; tile += npairs, ++local) {
        const int slot = local % INFO_RING;
        if (!mbar_wait(&info_empty[slot], ((local / INFO_RING) & 1u) ^ 1u, abort_flag, P.status)) break;
        const TileCoord c = decode_tile(P, tile, &seg);
        const Problem& pr = P.prob[c.p];
        float alpha = pr.alpha, beta = pr.beta;
        if (PS && pr.scale_part) {
          if (pr.scale != sc_part || c.b != sc_b) {
            // 1 / (||X_b||_F + eps) from the matrix's 32 partial sums, added by a fixed pairwise
            // tree in fp32 (fp64 arithmetic on this lane stalls the C loader and publishing lanes
            // of its warp); in fp64 only when the fp32 sum overflows
            const float4* pp = reinterpret_cast<const float4*>(pr.scale + (long long)c.b * SCALE_NPART);
            float4 v[SCALE_NPART / 4];
#pragma unroll
            for (int q = 0; q < SCALE_NPART / 4; ++q) v[q] = pp[q];
            float u[SCALE_NPART / 4];
#pragma unroll
            for (int q = 0; q < SCALE_NPART / 4; ++q) u[q] = (v[q].x + v[q].y) + (v[q].z + v[q].w);
#pragma unroll
            for (int w = SCALE_NPART / 8; w >= 1; w /= 2)
#pragma unroll
              for (int q = 0; q < w; ++q) u[q] = u[2 * q] + u[2 * q + 1];
            const float t = u[0];
            if (t <= 3.0e38f) {
              sc_last = __fdiv_rn(1.f, __fadd_rn(__fsqrt_rn(t), P.scale_eps));
            } else {
              double d = 0.0;
#pragma unroll
              for (int q = 0; q < SCALE_NPART / 4; ++q) d += ((double)v[q].x + v[q].y) + ((double)v[q].z + v[q].w);
              sc_last = (float)(1.0 / (sqrt(d) + (double)P.scale_eps));
            }
            sc_part = pr.scale;
            sc_b = c.b;
          }
          alpha *= powi(sc_last, pr.alpha_pow);
          beta *= powi(sc_last, pr.beta_pow);
        } else if (pr.scale) {
          const float sc = pr.scale[c.b];
          alpha *= powi(sc, pr.alpha_pow);
          beta *= powi(sc, pr.beta_pow);
        }
        uint32_t pf = (uint32_t)c.p;
        if (pr.has_c) pf |= TI_HAS_C;
        if (pr.sym && c.I != c.J && pr.mirror_out) pf |= TI_MIRROR;
        if (pr.has_d2 && c.I == c.J) pf |= TI_DIAG;
        if (pr.c_trans) pf |= TI_C_TRANS;
        if (pr.c_f16) pf |= TI_C_F16;
        if (pr.d_trans) pf |= TI_D_TRANS;
        if (pr.d_f16) pf |= TI_D_F16;
        if (pr.check_finite) pf |= TI_CHECK;
        if (pr.has_d2) pf |= TI_HAS_D2;
        if (pr.publish) pf |= TI_PUBLISH;
        if (c.p == P.rmo.prob) pf |= TI_ROWMAP;
        pf |= (uint32_t)(pr.d_trans ? 1 : pr.d_mode) << TI_DMODE_SHIFT;
        TileInfo& e = info[slot];
        e.pf = pf;
        e.b = c.b;
        e.ij = (uint32_t)c.I | ((uint32_t)c.J << 16);
        e.ctr_off = pr.ctr_off;
        e.alpha = alpha;
        e.beta = beta;
        e.gamma = pr.gamma;
        e.diag_limit = pr.diag_limit;
        e.kblocks = pr.kblocks;
        e.kf = (pr.a_mn ? KF_A_MN : 0u) | (pr.b_mn ? KF_B_MN : 0u) | (pr.a_upper ? KF_A_UPPER : 0u) |
               (pr.b_upper ? KF_B_UPPER : 0u) | (pr.ab_f16 ? KF_AB_F16 : 0u) | (pr.dep_mask ? KF_DEP : 0u) |
               ((uint32_t)pr.c_mode << KF_CMODE_SHIFT);
        mbar_arrive(&info_full[slot]);  // release: the entry is visible to the epilogue's wait
      }
    }
    if (lane == 3) {
      // ---------------- publishing lane (both CTAs) ----------------
      // Publishes each tile's completion to the dependent tiles once the epilogue has seen its
      // stores land: the release at GPU scope waits for the CTA's earlier writes to become
      // visible device-wide, which kept every epilogue thread waiting at the tile's last
      // barrier when the storing thread did it itself.
      int local = 0;
      for (int tile = pair; tile < P.total_tiles; tile += npairs, ++local) {
        const int slot = local % INFO_RING;
        const uint32_t ph = (local / INFO_RING) & 1u;
        if (!mbar_wait(&info_full[slot], ph, abort_flag, P.status)) break;
        const uint32_t pf = info[slot].pf;
        const int ctr = info[slot].ctr_off + info[slot].b;
        if (!mbar_wait(&info_stored[slot], ph, abort_flag, P.status)) break;
        if (pf & TI_PUBLISH) red_release_gpu_add(P.counters + ctr, 1);
        mbar_arrive(&info_empty[slot]);
      }
    }
    if (lane == 0) {
      // ---------------- C-tile loader (both CTAs) ----------------
      // Loads the C chunks of the next tile as soon as the epilogue releases each buffer,
      // a whole main loop ahead of their use.
      uint32_t qc = 0;  // C chunks loaded so far (ring slot and phase)
      int local = 0;
      for (int tile = pair; tile < P.total_tiles; tile += npairs, ++local) {
        const int islot = local % INFO_RING;
        if (!mbar_wait(&info_full[islot], (local / INFO_RING) & 1u, abort_flag, P.status)) break;
        const TileHead h = tile_head(&info[islot], Geo<CG>::KSH);
        if (!(h.pf & TI_HAS_C)) continue;
        const TileCoord c = h.c;
        const Problem& pr = P.prob[c.p];  // (tensor-map address only)
        const int m0 = c.I * TT + (int)rank * TM;
        const int n0 = c.J * TT;
        if ((h.kf & KF_DEP) && !wait_ready(ready_tile, tile, abort_flag, P.status)) break;
        bool ok = true;
        const CUtensorMap* const tmC = &pr.tmC;
        const int c_mode = (int)((h.kf >> KF_CMODE_SHIFT) & 3u);
        for (int ch = 0; ch < NCHUNK; ++ch, ++qc) {
          const uint32_t q = qc % C_BUFS;
          if (!mbar_wait(&cempty[q], ((qc / C_BUFS) & 1u) ^ 1u, abort_flag, P.status)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&cfull[q], CHUNK_BYTES);
          chunk_load(SC + q * CHUNK_BYTES, tmC, &cfull[q], c_mode, m0, n0 + ch * CHUNK, c.b);
        }
        if (!ok) break;
      }
    }
  } else if (warp < PROD2_WARP) {
    // ---------------- epilogue (warps 3..10 of both CTAs) ----------------
    const int et = threadIdx.x - 32 * FIRST_EPI_WARP;
    const int ew = warp - FIRST_EPI_WARP;
    const int quarter = warp & 3;  // TMEM lanes this warp may read
    const int half = ew >> 2;      // which 32 of a chunk's 64 columns
    const int r = quarter * 32 + lane;
    // the accumulator barriers the epilogue releases: the leader's for a CTA pair
    const uint32_t tempty_leader0 = CG == 2 ? mapa_shared(smem_u32(&tempty[0]), 0) : smem_u32(&tempty[0]);
    const uint32_t tempty_leader1 = CG == 2 ? mapa_shared(smem_u32(&tempty[1]), 0) : smem_u32(&tempty[1]);
    uint32_t qc = 0;  // C chunks consumed so far (ring slot and phase)
    uint32_t gc = 0;  // chunks stored so far (output staging buffers)
    // Row-mapped outputs: the W row of each of a tile's rows (-1 past the valid product rows)
    // is written to the tile's row buffer during the previous tile's first chunk (its map entry
    // loaded at that tile's start), and the tile's first chunk of W rows is loaded into cvec at
    // the previous tile's end, so that neither wait is on the tile's own path.
    int* const rm_idx_all = reinterpret_cast<int*>(smem + OFF_BAR + RM_IDX_OFF);  // [2][TM]
    const int rm_cols = P.rmo.cols, rm_has_c = P.rmo.has_c;
    auto rm_row = [&](const TileInfo& e, int i) {
      const int prow = (int)(e.ij & 0xFFFFu) * TT + (int)rank * TM + i;
      return prow < P.rmo.rows ? P.rmo.map[(long long)e.b * P.rmo.map_stride + prow] : -1;
    };
    auto rm_base = [&](const TileInfo& e) {
      return static_cast<const uint16_t*>(P.rmo.ptr) + (long long)e.b * P.rmo.stride;
    };
    uint4 cvec[4];  // this thread's row segment of the next row-mapped chunk's W
    if (pair < P.total_tiles) {
      if (et == 0) *epi_flag = mbar_wait(&info_full[0], 0u, abort_flag, P.status) ? 1 : 0;
      named_bar_sync(1, EPI_THREADS);
      if (*epi_flag && (info[0].pf & TI_ROWMAP)) {
        if (et < TM) rm_idx_all[et] = rm_row(info[0], et);
        named_bar_sync(1, EPI_THREADS);
        if (rm_has_c)
          rowmap_own_load(cvec, rm_base(info[0]), P.rmo.ld, rm_idx_all[r], (int)(info[0].ij >> 16) * TT + half * 32,
                          rm_cols);
      }
    }
    int local = 0;
    for (int tile = pair; tile < P.total_tiles; tile += npairs, ++local) {
      const int acc = local & 1;
      const uint32_t aph = (local >> 1) & 1;
      const int islot = local % INFO_RING, nslot = (local + 1) % INFO_RING;
      const bool has_next = tile + npairs < P.total_tiles;
      // the tile's parameters and the next tile's (decoded ahead by the tile-info lane), then
      // the accumulator; before a row-mapped tile's staging, every TMA store has read its buffer
      if (et == 0) {
        bool okw = mbar_wait(&info_full[islot], (local / INFO_RING) & 1u, abort_flag, P.status);
        if (okw && has_next) okw = mbar_wait(&info_full[nslot], ((local + 1) / INFO_RING) & 1u, abort_flag, P.status);
        if (okw) okw = mbar_wait(&tfull[acc], aph, abort_flag, P.status);
        if (okw && (info[islot].pf & TI_ROWMAP)) bulk_wait_read<0>();
        *epi_flag = okw ? 1 : 0;
      }
      named_bar_sync(1, EPI_THREADS);
      if (!*epi_flag) break;
      TileCoord c;
      const TileInfo ti = info[islot];
      c.p = (int)(ti.pf & 0xFFu);
      c.b = ti.b;
      c.I = (int)(ti.ij & 0xFFFFu);
      c.J = (int)(ti.ij >> 16);
      const Problem& pr = P.prob[c.p];
      const float alpha = ti.alpha, beta = ti.beta;
      const bool has_c = (ti.pf & TI_HAS_C) != 0;
      const bool mirror = (ti.pf & TI_MIRROR) != 0;
      const bool want_diag = (ti.pf & TI_DIAG) != 0;
      // per-product fields used inside the chunk loop, in registers (see KLoop)
      const int c_trans = (ti.pf & TI_C_TRANS) != 0, c_f16 = (ti.pf & TI_C_F16) != 0;
      const int d_trans = (ti.pf & TI_D_TRANS) != 0, d_f16 = (ti.pf & TI_D_F16) != 0;
      const int d_mode = (int)((ti.pf >> TI_DMODE_SHIFT) & 3u);
      const int check_finite = (ti.pf & TI_CHECK) != 0, has_d2 = (ti.pf & TI_HAS_D2) != 0;
      const int diag_limit = ti.diag_limit;
      const bool publish = (ti.pf & TI_PUBLISH) != 0;
      const float gamma = ti.gamma;
      const int m0 = c.I * TT + (int)rank * TM;  // first row of this CTA's half
      const int n0 = c.J * TT;
      const bool rowmap = (ti.pf & TI_ROWMAP) != 0;
      const int* const rows_mine = rm_idx_all + (local & 1) * TM;
      int* const rows_next = rm_idx_all + ((local + 1) & 1) * TM;
      const bool next_rowmap = has_next && (info[nslot].pf & TI_ROWMAP) != 0;
      const TileInfo* const nti = &info[nslot];
      int next_row = -1;  // (its map entry: the load's latency passes under this tile's first chunk)
      if (next_rowmap && et < TM) next_row = rm_row(*nti, et);
      tc_fence_after();
      const int diag_col = (int)rank * TM + r;  // tile column of this row's diagonal element
      const bool diag_mine = want_diag && ((diag_col >> 5) & 1) == half;
      float dv = 0.f;
      bool bad = false;
      if (rowmap) {
        // per chunk: W rows staged in shared memory by whole-row 16-byte loads, every thread
        // updates its own row segment there (fp32, one rounding), whole-row stores back to W
        const uint16_t* const base_mine = rm_base(ti);
        const int wr_mine = rows_mine[r];  // this thread's W row
        for (int ch = 0; ch < NCHUNK; ++ch, ++gc) {
          // chunks alternate between the two staging buffers, so that a chunk's staging does not
          // wait for the previous chunk's stores to have read theirs
          uint8_t* const sd = SD + (gc % OUT_BUFS) * CHUNK_BYTES;
          const int col0 = n0 + ch * CHUNK;
          if (ch == 0 && next_rowmap && et < TM) rows_next[et] = next_row;
          uint32_t v[32];
          __syncwarp();
          tmem_ld_32x32b_x32(tmem_base + acc * TT + ch * CHUNK + half * 32 + ((uint32_t)(quarter * 32) << 16), v);
          tmem_ld_wait();
          if (ch == NCHUNK - 1) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) acc_release<CG>(acc ? tempty_leader1 : tempty_leader0);
          }
          float2 o[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) o[i] = make_float2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
          if (alpha != 1.f) {
            const float2 a2 = make_float2(alpha, alpha);
#pragma unroll
            for (int i = 0; i < 16; ++i) o[i] = __fmul2_rn(a2, o[i]);
          }
          if (rm_has_c) {
            uint32_t cw[16];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              cw[4 * q] = cvec[q].x;
              cw[4 * q + 1] = cvec[q].y;
              cw[4 * q + 2] = cvec[q].z;
              cw[4 * q + 3] = cvec[q].w;
            }
            axpy_h16x2(o, cw, beta, d_f16);
            // the next chunk's (or the next row-mapped tile's first chunk's) segment
            if (ch + 1 < NCHUNK)
              rowmap_own_load(cvec, base_mine, P.rmo.ld, wr_mine, col0 + CHUNK + half * 32, rm_cols);
            else if (next_rowmap)
              rowmap_own_load(cvec, rm_base(*nti), P.rmo.ld, rows_next[r], (int)(nti->ij >> 16) * TT + half * 32,
                              rm_cols);
          }
          if (check_finite) {
            float2 z = make_float2(0.f, 0.f);
#pragma unroll
            for (int i = 0; i < 16; ++i) z = __ffma2_rn(o[i], make_float2(0.f, 0.f), z);
            bad |= !(z.x == 0.f && z.y == 0.f);
          }
          uint32_t pk[16];
          pack_h16x2(o, pk, d_f16);
          // each thread overwrites exactly the values it read
#pragma unroll
          for (int q = 0; q < 4; ++q)
            *reinterpret_cast<uint4*>(sd + off_direct(r, half * 32 + q * 8)) =
                make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
          named_bar_sync(1, EPI_THREADS);
          rowmap_chunk_store(sd, P.rmo.ptr, (long long)c.b * P.rmo.stride, P.rmo.ld, rows_mine, et, col0, rm_cols);
          // (the buffer is staged again two chunks on, after every thread has passed the next
          // chunk's barriers, and so finished these stores)
        }
        if (publish) {
          // the tile's stores are visible before its completion is published
          __threadfence();
          named_bar_sync(1, EPI_THREADS);
        }
      }
      for (int ch = 0; ch < (rowmap ? 0 : NCHUNK); ++ch, ++gc) {
        uint8_t* sd = SD + (gc % OUT_BUFS) * CHUNK_BYTES;
        uint32_t v[32];
        __syncwarp();
        tmem_ld_32x32b_x32(tmem_base + acc * TT + ch * CHUNK + half * 32 + ((uint32_t)(quarter * 32) << 16), v);
        tmem_ld_wait();
        if (ch == NCHUNK - 1) {
          // the accumulator has been read: release it to the leader's MMA issuer
          tc_fence_before();
          __syncwarp();
          if (lane == 0) acc_release<CG>(acc ? tempty_leader1 : tempty_leader0);
        }
        float2 o[16];  // the row's 32 values, in pairs
#pragma unroll
        for (int i = 0; i < 16; ++i) o[i] = make_float2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
        if (alpha != 1.f) {
          const float2 a2 = make_float2(alpha, alpha);
#pragma unroll
          for (int i = 0; i < 16; ++i) o[i] = __fmul2_rn(a2, o[i]);
        }
        if (has_c) {
          const uint32_t q = qc % C_BUFS;
          const uint8_t* sc = SC + q * CHUNK_BYTES;
          if (!mbar_wait(&cfull[q], (qc / C_BUFS) & 1u, abort_flag, P.status)) *epi_flag = 0;
          uint32_t cw[16];  // the row's 32 C values, two per word
          if (!c_trans) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const uint4 w = *reinterpret_cast<const uint4*>(sc + off_direct(r, half * 32 + q * 8));
              cw[4 * q] = w.x;
              cw[4 * q + 1] = w.y;
              cw[4 * q + 2] = w.z;
              cw[4 * q + 3] = w.w;
            }
          } else {
#pragma unroll
            for (int i = 0; i < 16; ++i)
              cw[i] = (uint32_t)*reinterpret_cast<const uint16_t*>(sc + off_trans(r, half * 32 + 2 * i)) |
                      ((uint32_t)*reinterpret_cast<const uint16_t*>(sc + off_trans(r, half * 32 + 2 * i + 1)) << 16);
          }
          axpy_h16x2(o, cw, beta, c_f16);
          __syncwarp();
          if (lane == 0) mbar_arrive(&cempty[q]);
          ++qc;
        }
        if (check_finite) {
          // x * 0 is 0 for every finite x and NaN for Inf / NaN: one paired FMA per two values
          float2 z = make_float2(0.f, 0.f);
#pragma unroll
          for (int i = 0; i < 16; ++i) z = __ffma2_rn(o[i], make_float2(0.f, 0.f), z);
          bad |= !(z.x == 0.f && z.y == 0.f);
        }
        if (diag_mine && (diag_col >> 6) == ch) {
          const int dj = diag_col & 31;
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            if (2 * i == dj) dv = o[i].x;
            if (2 * i + 1 == dj) dv = o[i].y;
          }
        }
        uint32_t pk[16];  // the row's 32 outputs rounded once, two per word
        pack_h16x2(o, pk, d_f16);
        // the stores that last read the staging buffer are done (waited for only now, so that
        // they drain while this chunk is loaded from tensor memory and computed)
        if (et == 0) {
          if (OUT_BUFS == 2) bulk_wait_read<1>(); else bulk_wait_read<0>();
        }
        if (ch == 0 && next_rowmap && et < TM) rows_next[et] = next_row;
        named_bar_sync(1, EPI_THREADS);
        if (!d_trans) {
#pragma unroll
          for (int q = 0; q < 4; ++q)
            *reinterpret_cast<uint4*>(sd + off_direct(r, half * 32 + q * 8)) =
                make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j)
            *reinterpret_cast<uint16_t*>(sd + off_trans(r, half * 32 + j)) = (uint16_t)(pk[j >> 1] >> (16 * (j & 1)));
        }
        fence_proxy_async_smem();
        named_bar_sync(1, EPI_THREADS);
        const int col0 = n0 + ch * CHUNK;
        const bool chunk_has_diag = want_diag && (ch == 2 * (int)rank || ch == 2 * (int)rank + 1);
        if (et == 0) {
          chunk_store(sd, &pr.tmD, d_mode, m0, col0, c.b);
          if (has_d2 && !chunk_has_diag) chunk_store(sd, &pr.tmD2, d_mode, m0, col0, c.b);
          bulk_commit();
        }
        if (mirror) {
          // the transposed copy goes through the same staging buffer once the stores above
          // have read it (mirrored tiles are never diagonal ones)
          if (et == 0) bulk_wait_read<0>();
          named_bar_sync(1, EPI_THREADS);
#pragma unroll
          for (int j = 0; j < 32; ++j)
            *reinterpret_cast<uint16_t*>(sd + off_trans(r, half * 32 + j)) = (uint16_t)(pk[j >> 1] >> (16 * (j & 1)));
          fence_proxy_async_smem();
          named_bar_sync(1, EPI_THREADS);
          if (et == 0) {
            chunk_store(sd, &pr.tmD, 1, m0, col0, c.b);
            if (has_d2) chunk_store(sd, &pr.tmD2, 1, m0, col0, c.b);
            bulk_commit();
          }
        }
        if (chunk_has_diag) {
          // D2 = D + gamma I: patch the diagonal with the fp32 value plus gamma, rounded once
          // (appendix B.2.3: adding a_t I to an already rounded Z loses a_t's precision)
          if (et == 0) bulk_wait_read<0>();
          named_bar_sync(1, EPI_THREADS);
          if (diag_mine && (diag_col >> 6) == ch && m0 + r < diag_limit)
            *reinterpret_cast<uint16_t*>(sd + off_direct(r, diag_col & 63)) = f_to_h16(dv + gamma, d_f16);
          fence_proxy_async_smem();
          named_bar_sync(1, EPI_THREADS);
          if (et == 0) {
            chunk_store(sd, &pr.tmD2, d_mode, m0, col0, c.b);
            bulk_commit();
          }
        }
      }
      // a row-mapped next tile's first chunk of W rows (a row-mapped tile issued it in its
      // last chunk)
      if (!rowmap && next_rowmap && rm_has_c)
        rowmap_own_load(cvec, rm_base(*nti), P.rmo.ld, rows_next[r], (int)(nti->ij >> 16) * TT + half * 32, rm_cols);
      if (bad) set_status(P.status, GNS_DEVST_NONFINITE);
      if (et == 0) {
        // this CTA's half of the tile is in global memory (products nothing in the launch
        // depends on skip the wait): the publishing lane announces it to dependent tiles
        if (publish) {
          bulk_wait_all();
          fence_proxy_async_global();
        }
        mbar_arrive(&info_stored[islot]);
      }
      named_bar_sync(1, EPI_THREADS);
      if (et == 0) mbar_arrive(&info_empty[islot]);  // every thread has read the tile's entry
      if (!*epi_flag) break;
    }
    if (et == 0) bulk_wait_all();
  }

  // lanes 1-31 of the producer and MMA warps wait here for lane 0 (aligned barriers below)
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if constexpr (CG == 2) cluster_sync_all();  // no remote arrival or peer MMA can still target this CTA
  if (warp == 1) {
    tc_fence_after();
    if constexpr (CG == 2)
      tmem_dealloc2(tmem_base, TMEM_COLS);
    else
      tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

}  // namespace tc

// ------------------------------------------------------------------------------------
// host side

static PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn(std::string* err) {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  if (!fn && err) *err = "cuTensorMapEncodeTiled is not available from the CUDA driver";
  return fn;
}

// 3-D tensor map of 16-bit elements (fp16 when f16, else bf16) over a batch of row-major
// matrices: dims {cols, rows, batch}, box {64, box_rows, 1}, 128-byte swizzle, zero fill out
// of bounds.
static bool encode_map(CUtensorMap* map, const MatRef& m, int64_t batch, int box_rows, int f16, std::string* err) {
  auto fn = get_encode_fn(err);
  if (!fn) return false;
  const int64_t ld_b = m.ld * 2;
  int64_t st_b = (batch > 1 ? m.stride : m.rows * m.ld) * 2;
  st_b = (st_b + 15) / 16 * 16;
  if (st_b == 0) st_b = 16;
  cuuint64_t dims[3] = {(cuuint64_t)m.cols, (cuuint64_t)m.rows, (cuuint64_t)batch};
  cuuint64_t strides[2] = {(cuuint64_t)ld_b, (cuuint64_t)st_b};
  cuuint32_t box[3] = {64u, (cuuint32_t)box_rows, 1u};
  cuuint32_t estr[3] = {1u, 1u, 1u};
  CUresult r = fn(map, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, m.ptr, dims,
                  strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    if (err) *err = "cuTensorMapEncodeTiled failed (code " + std::to_string((int)r) + ")";
    return false;
  }
  return true;
}

int device_sm_count() {
  static int cached[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) dev = 0;
  if (!cached[dev]) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    cached[dev] = n > 0 ? n : 1;
  }
  return cached[dev];
}

// Number of CTA groups (pairs for CG = 2, single CTAs for CG = 1) of the GEMM kernel that can
// be resident at once, and the one-time shared-memory opt-in. A persistent launch never asks
// for more: its groups wait on one another's completion counters.
template <class L, int CG, bool PS>
static int resident_groups(std::string* err) {
  static int cached[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) dev = 0;
  if (cached[dev]) return cached[dev];
  cudaError_t e =
      cudaFuncSetAttribute(tc::gemm_kernel<L, CG, PS>, cudaFuncAttributeMaxDynamicSharedMemorySize, L::SMEM_BYTES);
  if (e != cudaSuccess) {
    *err = std::string("cudaFuncSetAttribute: ") + cudaGetErrorString(e);
    return 0;
  }
  int groups = 0;
  if constexpr (CG == 2) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(2 * (device_sm_count() / 2), 1, 1);
    cfg.blockDim = dim3(tc::NUM_THREADS, 1, 1);
    cfg.dynamicSmemBytes = L::SMEM_BYTES;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaOccupancyMaxActiveClusters(&groups, tc::gemm_kernel<L, CG, PS>, &cfg);
    if (e != cudaSuccess || groups < 1) {
      (void)cudaGetLastError();
      groups = device_sm_count() / 2;
    }
  } else {
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, tc::gemm_kernel<L, CG, PS>, tc::NUM_THREADS,
                                                      L::SMEM_BYTES);
    if (e != cudaSuccess || per_sm < 1) {
      (void)cudaGetLastError();
      per_sm = 1;
    }
    groups = per_sm * device_sm_count();
  }
  cached[dev] = groups;
  return groups;
}

struct Segment {
  int p;
  int64_t b0, nb;
};

// Order of the tiles of one launch. Independent products (no dependency masks), or products
// over batches of different sizes, run problem after problem. A program of dependent
// products over one batch of B matrices runs in waves of W matrices: segment (w, p) holds
// the tiles of problem p for the matrices of wave w and is placed by the key p + D * w (ties
// to the lower wave). D = 0 is stage-major across the waves (W = B: every stage over the
// whole batch before the next one); D = nops runs wave after wave, every stage of a few
// matrices at a time, whose n x n buffers then stay in L2; values in between overlap the
// late stages of one wave with the early ones of the next. Every segment comes after the
// segments of earlier problems for the same matrices, so each tile depends only on earlier
// tiles. GNS_TILE_ORDER="W,D" in the environment overrides the default (a tuning knob).
static void tile_order(const GemmOp* ops, int nops, bool dependent, std::vector<Segment>* out) {
  out->clear();
  bool same = true;
  for (int i = 1; i < nops; ++i) same = same && ops[i].batch == ops[0].batch;
  const int64_t B = ops[0].batch;
  int64_t W = B;
  int64_t D = 0;
  if (dependent && same) {
    const char* env = getenv("GNS_TILE_ORDER");
    long w = 0, d = 0;
    if (env && sscanf(env, "%ld,%ld", &w, &d) == 2 && w > 0 && d >= 0) {
      W = std::min<int64_t>(w, B);
      D = d;
    }
    // the segment list must fit the launch parameters
    const int64_t max_waves = std::max<int64_t>(1, tc::MAX_SEG / nops);
    if ((B + W - 1) / W > max_waves) W = (B + max_waves - 1) / max_waves;
  }
  if (!dependent || !same) {
    for (int p = 0; p < nops; ++p) out->push_back({p, 0, ops[p].batch});
    return;
  }
  const int64_t nw = (B + W - 1) / W;
  struct Key {
    int64_t key, w;
    int p;
  };
  std::vector<Key> keys;
  for (int64_t w = 0; w < nw; ++w)
    for (int p = 0; p < nops; ++p) keys.push_back({p + D * w, w, p});
  std::stable_sort(keys.begin(), keys.end(), [](const Key& a, const Key& b) {
    return a.key != b.key ? a.key < b.key : a.w < b.w;
  });
  for (const Key& k : keys) out->push_back({k.p, k.w * W, std::min(W, B - k.w * W)});
}

int gemm_launch_tc(const GemmOp* ops, int nops, const uint32_t* dep_masks, int* counters, int32_t* dev_status,
                   void* stream, std::string* err, bool counters_zeroed) {
  using namespace tc;
  static_assert(sizeof(Params) <= 32764, "kernel parameter space");
  if (nops < 1 || nops > MAX_PROB) {
    *err = "internal: bad number of products in one launch";
    return GNS_ERR_INVALID;
  }
  // CTA-group size: single CTAs with 128 x 128 tiles when every product has at most 128
  // rows (GNS_CTA_GROUP=1 or 2 in the environment overrides, a tuning knob)
  int64_t max_m = 0, sym_pair_tiles = 0;
  for (int i = 0; i < nops; ++i) {
    max_m = std::max<int64_t>(max_m, ops[i].M);
    if (ops[i].sym) {
      const int64_t t = (ops[i].M + 255) / 256;
      sym_pair_tiles = std::max<int64_t>(sym_pair_tiles, ops[i].batch * t * (t + 1) / 2);
    }
  }
  // 1-CTA 128 x 128 tiles for products of at most 256 rows (a 256 x 256 tile of an n = 256
  // product has 4 K slices), and for small batches of n <= 1024 whose largest symmetric stage
  // has at most 48 pair tiles, which would leave most of the chip's 76 CTA pairs idle
  // (measured: 1-4 matrices of 1024 x 4096 and 16 of 512 x 2048 run 3-13 % faster on 1-CTA
  // tiles, 8 or more of 1024 x 4096 10-40 % slower)
  int cg = max_m <= 256 || (max_m <= 1024 && sym_pair_tiles > 0 && sym_pair_tiles <= 48) ? 1 : 2;
  if (const char* env = getenv("GNS_CTA_GROUP")) {
    if (env[0] == '1' && env[1] == 0) cg = 1;
    if (env[0] == '2' && env[1] == 0) cg = 2;
  }
  const int tile = 128 * cg;
  Params P;
  memset(&P, 0, sizeof(P));
  int tiles = 0;
  P.rmo.prob = -1;
  bool have_eps = false;  // a problem forms its scale from partial sums (their eps)
  for (int i = 0; i < nops; ++i) {
    const GemmOp& o = ops[i];
    Problem& pr = P.prob[i];
    if (o.row_map) {
      if (P.rmo.prob >= 0 || o.sym || o.d_trans || o.c_trans || o.D2.ptr || (o.C.ptr && o.C.ptr != o.D.ptr) ||
          o.D.ld % 8 || reinterpret_cast<uintptr_t>(o.D.ptr) % 16 || (o.batch > 1 && o.D.stride % 8)) {
        *err = "internal: unsupported row-mapped output";
        return GNS_ERR_INVALID;
      }
      P.rmo.prob = i;
      P.rmo.map = o.row_map;
      P.rmo.map_stride = (int)o.row_map_stride;
      P.rmo.ptr = o.D.ptr;
      P.rmo.ld = o.D.ld;
      P.rmo.stride = o.D.stride;
      P.rmo.rows = (int)o.M;
      P.rmo.cols = (int)o.N;
      P.rmo.has_c = o.C.ptr != nullptr && o.beta != 0.f;
    }
    const int dts[3] = {o.ab_dt, o.c_dt, o.d_dt};
    for (int t : dts)
      if (t != GNS_BF16 && t != GNS_F16) {
        *err = "internal: the tensor-core GEMM takes bf16 or fp16 matrices";
        return GNS_ERR_INVALID;
      }
    pr.ab_f16 = o.ab_dt == GNS_F16;
    pr.c_f16 = o.c_dt == GNS_F16;
    pr.d_f16 = o.d_dt == GNS_F16;
    if (!encode_map(&pr.tmA, o.A, o.batch, o.a_mn ? 64 : 128, pr.ab_f16, err)) return GNS_ERR_CUDA;
    if (!encode_map(&pr.tmB, o.B, o.batch, o.b_mn ? 64 : 128, pr.ab_f16, err)) return GNS_ERR_CUDA;
    pr.a_upper = o.a_upper;
    pr.b_upper = o.b_upper;
    pr.mirror_out = o.upper_out ? 0 : 1;
    if (o.a_upper && !encode_map(&pr.tmA2, o.A, o.batch, o.a_mn ? 128 : 64, pr.ab_f16, err)) return GNS_ERR_CUDA;
    if (o.b_upper && !encode_map(&pr.tmB2, o.B, o.batch, o.b_mn ? 128 : 64, pr.ab_f16, err)) return GNS_ERR_CUDA;
    // a row-mapped output reads its C in the epilogue: the C loader skips the problem
    pr.has_c = o.C.ptr != nullptr && o.beta != 0.f && !o.row_map;
    // one 128-row box per chunk where a map serves only direct chunks
    pr.c_mode = o.c_trans ? 1 : 2;
    const bool d_one_box = !o.d_trans && !(o.sym && !o.upper_out);
    pr.d_mode = d_one_box ? 2 : 0;
    if (pr.has_c && !encode_map(&pr.tmC, o.C, o.batch, o.c_trans ? 64 : 128, pr.c_f16, err)) return GNS_ERR_CUDA;
    if (!o.row_map && !encode_map(&pr.tmD, o.D, o.batch, d_one_box ? 128 : 64, pr.d_f16, err)) return GNS_ERR_CUDA;
    pr.has_d2 = o.D2.ptr != nullptr;
    if (pr.has_d2 && !encode_map(&pr.tmD2, o.D2, o.batch, d_one_box ? 128 : 64, pr.d_f16, err)) return GNS_ERR_CUDA;
    pr.a_mn = o.a_mn;
    pr.b_mn = o.b_mn;
    pr.kblocks = (int)((o.K + TK - 1) / TK);
    pr.tiles_m = (int)((o.M + tile - 1) / tile);
    pr.tiles_n = (int)((o.N + tile - 1) / tile);
    if (pr.tiles_m > 65535 || pr.tiles_n > 65535) {  // tile coordinates travel as 16-bit fields
      *err = "a product of more than 65535 tiles along one dimension";
      return GNS_ERR_UNSUPPORTED;
    }
    pr.sym = o.sym;
    const long long tpm = o.sym ? (long long)pr.tiles_m * (pr.tiles_m + 1) / 2 : (long long)pr.tiles_m * pr.tiles_n;
    if (tpm * o.batch + tiles > (long long)INT32_MAX) {
      *err = "the products of one call have more than 2^31 output tiles";
      return GNS_ERR_UNSUPPORTED;
    }
    pr.tiles_per_mat = (int)tpm;
    tiles += pr.tiles_per_mat * (int)o.batch;
    pr.alpha = o.alpha;
    pr.beta = o.beta;
    pr.gamma = o.gamma;
    pr.alpha_pow = o.alpha_pow;
    pr.beta_pow = o.beta_pow;
    pr.scale = o.scale;
    if (o.scale_part) {
      if (o.scale_npart != SCALE_NPART || reinterpret_cast<uintptr_t>(o.scale_part) % 16 != 0 ||
          (have_eps && o.scale_eps != P.scale_eps)) {
        *err = "internal: a norm scale formed from other than 32 aligned partial sums per matrix, or with "
               "another eps than the launch's";
        return GNS_ERR_UNSUPPORTED;
      }
      pr.scale = o.scale_part;
      pr.scale_part = 1;
      P.scale_eps = o.scale_eps;
      have_eps = true;
    }
    pr.c_trans = o.c_trans;
    pr.d_trans = o.d_trans;
    pr.diag_limit = (int)o.diag_limit;
    pr.check_finite = o.check_finite;
    pr.dep_mask = dep_masks ? dep_masks[i] : 0u;
    if (pr.dep_mask && !counters) {
      *err = "internal: dependent products need completion counters";
      return GNS_ERR_INVALID;
    }
    pr.publish = 0;
    if (dep_masks && counters)
      for (int j = i + 1; j < nops; ++j)
        if (dep_masks[j] & (1u << i)) pr.publish = 1;
  }
  int off = 0;
  for (int i = 0; i < nops; ++i) {
    P.prob[i].ctr_off = off;
    off += (int)ops[i].batch;
  }
  // tile order: segments (problem, first matrix, matrices), see tile_order()
  {
    std::vector<Segment> segs;
    tile_order(ops, nops, dep_masks != nullptr, &segs);
    if (segs.empty() || (int)segs.size() > MAX_SEG) {
      *err = "internal: tile order does not fit the launch parameters";
      return GNS_ERR_INVALID;
    }
    int t = 0;
    for (size_t i = 0; i < segs.size(); ++i) {
      P.seg_pb[i] = ((uint32_t)segs[i].p << 24) | (uint32_t)segs[i].b0;
      P.seg_tile[i] = t;
      t += P.prob[segs[i].p].tiles_per_mat * (int)segs[i].nb;
    }
    P.nseg = (int)segs.size();
    if (t != tiles) {
      *err = "internal: tile order does not cover every tile once";
      return GNS_ERR_INVALID;
    }
  }
  P.nprob = nops;
  P.total_tiles = tiles;
  P.status = dev_status;
  P.counters = counters;
  if (counters && tiles > 0 && !counters_zeroed) {
    cudaError_t me = cudaMemsetAsync(counters, 0, sizeof(int) * off, static_cast<cudaStream_t>(stream));
    if (me != cudaSuccess) {
      *err = std::string("counter reset: ") + cudaGetErrorString(me);
      return GNS_ERR_CUDA;
    }
  }
  if (tiles == 0) return GNS_OK;
  long long slices = 0;  // K slices over all tiles of the launch
  int64_t max_batch = 0;
  for (int i = 0; i < nops; ++i) {
    slices += (long long)P.prob[i].kblocks * P.prob[i].tiles_per_mat * ops[i].batch;
    max_batch = std::max<int64_t>(max_batch, ops[i].batch);
  }
  const bool deep = slices <= (long long)DEEP_MAX_SLICES_PER_TILE * tiles ||
                    (max_batch <= DEEP_SMALL_BATCH && slices <= (long long)DEEP_MAX_SLICES_SMALL_BATCH * tiles);
  const bool ps = have_eps;
  const int resident = cg == 2 ? (deep ? (ps ? resident_groups<DeepPlan, 2, true>(err)
                                             : resident_groups<DeepPlan, 2, false>(err))
                                       : (ps ? resident_groups<ShallowPlan, 2, true>(err)
                                             : resident_groups<ShallowPlan, 2, false>(err)))
                               : (deep ? (ps ? resident_groups<DeepPlan, 1, true>(err)
                                             : resident_groups<DeepPlan, 1, false>(err))
                                       : (ps ? resident_groups<ShallowPlan, 1, true>(err)
                                             : resident_groups<ShallowPlan, 1, false>(err)));
  if (resident < 1) return GNS_ERR_CUDA;
  const int groups = std::min(tiles, resident);
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  // PS instances wait (grid_dep_wait) for the kernel ahead of them before they touch global
  // memory: only they are programmatic dependent launches
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = 2;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.gridDim = dim3(cg * groups, 1, 1);
  cfg.blockDim = dim3(NUM_THREADS, 1, 1);
  cfg.dynamicSmemBytes = deep ? DeepPlan::SMEM_BYTES : ShallowPlan::SMEM_BYTES;
  cfg.stream = static_cast<cudaStream_t>(stream);
  cfg.attrs = ps ? attr : attr + 1;
  cfg.numAttrs = (ps ? 1 : 0) + (cg == 2 ? 1 : 0);
  cudaError_t e;
  if (cg == 2) {
    if (deep)
      e = ps ? cudaLaunchKernelEx(&cfg, gemm_kernel<DeepPlan, 2, true>, P)
             : cudaLaunchKernelEx(&cfg, gemm_kernel<DeepPlan, 2, false>, P);
    else
      e = ps ? cudaLaunchKernelEx(&cfg, gemm_kernel<ShallowPlan, 2, true>, P)
             : cudaLaunchKernelEx(&cfg, gemm_kernel<ShallowPlan, 2, false>, P);
  } else {
    if (deep)
      e = ps ? cudaLaunchKernelEx(&cfg, gemm_kernel<DeepPlan, 1, true>, P)
             : cudaLaunchKernelEx(&cfg, gemm_kernel<DeepPlan, 1, false>, P);
    else
      e = ps ? cudaLaunchKernelEx(&cfg, gemm_kernel<ShallowPlan, 1, true>, P)
             : cudaLaunchKernelEx(&cfg, gemm_kernel<ShallowPlan, 1, false>, P);
  }
  if (e != cudaSuccess) {
    *err = std::string("tcgen05 GEMM launch: ") + cudaGetErrorString(e);
    return GNS_ERR_CUDA;
  }
  return GNS_OK;
}

}  // namespace gns
