// Gram Newton-Schulz (Dion3: Full-Stack Orthogonal Updates, sec. 4.2, Algorithm 3) and
// standard Newton-Schulz (Algorithm 1) for small matrices, sm_103a: one CTA carries one
// matrix's whole chain of products, with X and the n x n iterates held on chip.
//
// Scope: the oriented X is n x m with n <= 128 and m <= 512 (any coefficient schedule,
// any restarts). Every product of the chain is then one 128-row MMA group on one SM: the
// Gram product X X^T (K = m), the n x n products of an iteration (128 x 128 x 128) and
// Q X (128 x m x 128). Running them as tiles of the batched kernel costs a few microseconds
// of fixed work per tile (counters, stores, reloads) for a fraction of a microsecond of MMA;
// here nothing between the load of X and the store of the result leaves the SM:
//
//   shared memory  X (128 x 512 16-bit, 128 KiB; one TMA load per matrix, overwritten in
//                  place by X <- Q X), R, Z, Q (128 x 128, 32 KiB each), all in the
//                  128-byte-swizzled layout that the MMA reads: 64-column panels of 128 rows
//                  (a tall X arrives transposed: 64-row panels of its m rows, read MN-major);
//   tensor memory  four 128-column fp32 accumulators (all 512 columns; Q X takes all four);
//   warp 0         TMA loads of the next matrix's X once the last product has read the region;
//   warp 1         TMEM allocation and the MMA issuer (one thread);
//   warps 2-9      epilogue: thread = accumulator row, two warps per TMEM lane quarter, each
//                  taking every second 32-column group. Results go back into the swizzled
//                  operand buffers, in the product type, for the next MMA, or to global memory
//                  at the end.
//
// Products and epilogues follow a list of ops built on the host. An op's MMAs wait for the
// epilogue of the latest op that wrote one of its operands or used its accumulator columns;
// epilogues complete in list order, so one mbarrier wait covers every earlier epilogue.
// In-place updates (RZ over R, R_t over RZ, Q_t over Q, X <- Q X over X) are safe because an
// epilogue starts only after its own product, and with it every earlier product, completed.
// The Frobenius norm of X is summed from shared memory by the epilogue warps while the first
// Gram product runs, unless the caller passes it.
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "chain_small.h"
#include "common.cuh"

namespace gns {
namespace chain {

constexpr int NP = 128;                      // rows of X and of the n x n iterates (padded)
constexpr int MAXM = 512;                    // columns of X
constexpr int PANEL_BYTES = NP * 128;        // 128 rows x 64 16-bit columns
constexpr int NN_BYTES = 2 * PANEL_BYTES;    // one n x n iterate
constexpr int XREG_BYTES = NP * MAXM * 2;    // X
constexpr int MAX_OPS = 96;                  // 4 T + 2 (T - 1) + 2 at T = 16
constexpr int FIRST_EPI_WARP = 2;
#ifndef GNS_CHAIN_EPI_WARPS
#define GNS_CHAIN_EPI_WARPS 8
#endif
constexpr int EPI_WARPS = GNS_CHAIN_EPI_WARPS;  // a multiple of 4: EPI_WARPS / 4 per TMEM lane quarter
constexpr int NG = EPI_WARPS / 4;               // warps per lane quarter; each takes every NG-th 32-column group
constexpr int NUM_THREADS = 32 * (FIRST_EPI_WARP + EPI_WARPS);

// shared-memory plan (offsets from a 1024-byte-aligned base)
constexpr int OFF_R = XREG_BYTES;
constexpr int OFF_Z = OFF_R + NN_BYTES;
constexpr int OFF_Q = OFF_Z + NN_BYTES;
constexpr int OFF_BAR = OFF_Q + NN_BYTES;
constexpr int BAR_BYTES = 8 * (1 + 2 * MAX_OPS) + 16 + 4 * 2 * EPI_WARPS;
constexpr int SMEM_BYTES = 1024 + OFF_BAR + BAR_BYTES;
static_assert(SMEM_BYTES <= 232448, "shared memory budget");

// buffers
enum : uint8_t { BUF_R = 0, BUF_Z = 1, BUF_Q = 2, BUF_X = 3 };
// products: X X^T (K = m), n x n (A K-major, B MN-major), A X (n x m, K = n)
enum : uint8_t { K_GRAM = 0, K_NN = 1, K_AX = 2 };
// epilogues (acc = the fp32 accumulator, s = 1/(||X||_F + eps) where the op reads user X)
enum : uint8_t {
  E_SCALE = 0,  // d = s^2 acc                          (Gram products)
  E_POLY = 1,   // d = p1 acc + p0 c; Q = d + p2 I       (Z, or standard NS's b A + c A^2)
  E_AXPY = 2,   // d = acc + p0 c                        (RZ, R_t, Q_t)
  E_XSET = 3,   // X = s acc                             (restart: X <- Q X)
  E_XAXPY = 4,  // X = s (p0 X + acc)                    (standard NS: X <- a X + B X)
  E_OUT = 5     // D = alpha s (acc [+ p0 X]) + beta D   (the result)
};
// op flags
// F_XIN: the op reads the X region while it still holds the input as stored (a tall
// matrix's storage is X transposed: the products read it the other way)
enum : uint8_t { F_QINIT = 1, F_USER = 2, F_XIN = 4, F_ADDX = 8 };

struct Op {
  uint8_t kind, epi;
  uint8_t a, b;  // operand buffers (K_NN: A = a, B = b; K_AX: A = a, B = X; K_GRAM: X, X)
  uint8_t c, d;  // epilogue addend and output buffers
  uint8_t slot;  // first 128-column accumulator
  uint8_t flags;
  int16_t dep;   // wait for this op's epilogue before issuing (-1: none)
  int8_t half;   // K_AX: the half of the columns it computes (0 or 1), or -1: all
  uint8_t pad;
  float p0, p1, p2;
};

constexpr int MAX_GROUPS = 8;  // shape groups one launch carries

// One shape group of a launch: its matrices are the launch's matrices first .. first+count-1.
struct Group {
  CUtensorMap tmX;  // X: rows of the n x m operand (box 64 x 128), or a tall matrix's m x n
                    // storage (box 64 x 64); zero fill outside the matrix
  CUtensorMap tmD;  // the result, 32 x 32 boxes, 64-byte swizzle (used when d_tma)
  void* D;
  const float* inv;  // per-matrix 1/(||X||_F + eps) (norm_mode 1)
  long long ldd, sd;
  int first, count, n, m, mp;  // first: the group's first job of the launch; mp: m padded to 64
  int xt;                      // the input X is stored transposed (m x n)
  int pack, nb;                // matrices per 128-row chain (1, 2 or 4) and rows per block (128 / pack)
  int d_f16, d_trans, has_c;
  int d_tma;  // the result goes out by TMA stores (no addend to read)
  float alpha, beta;
};

struct Params {
  Group grp[MAX_GROUPS];
  Op ops[MAX_OPS];  // one list for every group (X <- Q X and Q X take all four accumulators)
  int nops, ngroups, total;
  int op0_prev;   // the last op of a matrix that uses accumulator 0: the next matrix's first
                  // product waits for its epilogue
  int ab_f16;     // products in fp16 (else bf16)
  int norm_mode;  // 0: s = 1; 1: s = inv[b]; 2: from the trace of the first Gram product
  int check_finite;
  float eps;
  int32_t* status;
};

// the group of launch matrix i (groups are in order of their first matrix)
__device__ __forceinline__ int group_of(const Params& P, int i) {
  int g = 0;
  while (g + 1 < P.ngroups && i >= P.grp[g + 1].first) ++g;
  return g;
}

__host__ __device__ inline uint32_t buf_off(int buf) {
  return buf == BUF_R ? OFF_R : buf == BUF_Z ? OFF_Z : buf == BUF_Q ? OFF_Q : 0u;
}

// byte offset of the 16-byte chunk j (columns 8j .. 8j+7) of row r in a 64-column panel
// (128-byte swizzle: chunk j of row r sits at position j ^ (r mod 8))
__device__ __forceinline__ uint32_t chunk_off(int r, int j) { return (uint32_t)(r * 128 + ((j ^ (r & 7)) << 4)); }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// 32 accumulator columns of this warp's lane quarter, starting at column col
__device__ __forceinline__ void load_acc32(uint32_t trow, int col, float (&v)[32]) {
  uint32_t u[32];
  tmem_ld_32x32b_x32(trow + (uint32_t)col, u);
  tmem_ld_wait();
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(u[i]);
}

// The columns of the first half of a split A X product: mp / 2 rounded up to a whole 64-column
// panel (the operand descriptors start on panel boundaries), at most 256 (one MMA).
__host__ __device__ __forceinline__ int ax_split(int mp) { return min(256, (mp / 2 + 63) & ~63); }

// ------------------------------------------------------------------------------------
// MMA issue (one thread). Descriptors: a K-major operand advances 32 bytes per K = 16 step
// inside its 64-column panel; an MN-major one advances 16 rows (2048 bytes), its 64-wide
// MN blocks lbo bytes apart.

__device__ __forceinline__ void issue_op(const Op o, int mp, int ab, bool xt_in, uint32_t s, uint32_t tmem) {
  const bool xt = xt_in && (o.flags & F_XIN) != 0;
  if (o.kind == K_GRAM) {
    // X X^T: A(i,k) = B(i,k) = X[i][k]
    const uint32_t d = tmem + 128u * o.slot;
    if (!xt) {
      const uint32_t idesc = idesc_f16kind_f32(128, 128, 0, 0, ab);
      for (int kb = 0; kb < mp / 64; ++kb)
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint64_t desc = sdesc_sw128(s + kb * PANEL_BYTES + kk * 32, 16, 1024);
          umma_f16kind(d, desc, desc, idesc, (kb | kk) != 0 ? 1u : 0u);
        }
    } else {
      // stored transposed: row k of the region holds X[0..63][k], the second 64 rows of X
      // one block of mp rows further
      const uint32_t idesc = idesc_f16kind_f32(128, 128, 1, 1, ab);
      for (int ks = 0; ks < mp / 16; ++ks) {
        const uint64_t desc = sdesc_sw128(s + ks * 2048, (uint32_t)(mp * 128), 1024);
        umma_f16kind(d, desc, desc, idesc, ks != 0 ? 1u : 0u);
      }
    }
  } else if (o.kind == K_NN) {
    // A (K-major) times B (MN-major): the product of the two stored matrices
    const uint32_t idesc = idesc_f16kind_f32(128, 128, 0, 1, ab);
    const uint32_t d = tmem + 128u * o.slot;
    const uint32_t A = s + buf_off(o.a), Bm = s + buf_off(o.b);
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      const uint64_t ad = sdesc_sw128(A + (ks >> 2) * PANEL_BYTES + (ks & 3) * 32, 16, 1024);
      const uint64_t bd = sdesc_sw128(Bm + ks * 2048, PANEL_BYTES, 1024);
      umma_f16kind(d, ad, bd, idesc, ks != 0 ? 1u : 0u);
    }
  } else {
    // A X, n x m: B(j,k) = X[k][j], MN-major from the row layout, K-major from the
    // transposed one. Columns [c0, c0 + N) go to TMEM columns from 256 hh: the whole
    // product in N = 256 pieces, or the op's half (the first ax_split(mp) columns, or the rest)
    const uint32_t A = s + buf_off(o.a);
    const int h0 = o.half < 0 ? 0 : o.half, h1 = o.half < 0 ? 2 : o.half + 1;
    for (int hh = h0; hh < h1; ++hh) {
      const int c0 = o.half < 0 ? 256 * hh : (hh == 0 ? 0 : ax_split(mp));
      const int N = o.half < 0 ? min(256, mp - c0) : (hh == 0 ? ax_split(mp) : mp - c0);
      if (N <= 0) continue;
      const uint32_t idesc = idesc_f16kind_f32(128, N, 0, xt ? 0 : 1, ab);
      const uint32_t d = tmem + 256u * hh;
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        const uint64_t ad = sdesc_sw128(A + (ks >> 2) * PANEL_BYTES + (ks & 3) * 32, 16, 1024);
        const uint64_t bd =
            xt ? sdesc_sw128(s + (ks >> 2) * (mp * 128) + (ks & 3) * 32 + c0 * 128, 16, 1024)
               : sdesc_sw128(s + (c0 / 64) * PANEL_BYTES + ks * 2048, PANEL_BYTES, 1024);
        umma_f16kind(d, ad, bd, idesc, ks != 0 ? 1u : 0u);
      }
    }
  }
}

// ------------------------------------------------------------------------------------
// epilogues: thread = accumulator row r (TMEM lane), g = the warp's 32-column group (columns
// 32g .. 32g+31 of an n x n product: chunks 4(g mod 2) .. +3 of panel g / 2). The launch
// parameters they use are copied into registers once (Ctx, by value), and each op into
// registers before its epilogue: read through references into the parameter space, every
// field would be reloaded after each shared-memory store the compiler cannot prove
// independent of it. The arithmetic runs on value pairs (the paired fp32 instructions, each
// element rounded as its scalar form would be) and is compiled once per 16-bit type: the
// epilogue is on the chain's critical path and bound by its instruction count.

struct Ctx {
  uint8_t* sm;
  uint32_t trow;
  int r, g, ew, lane, n, m, mp;
  int d_f16, d_trans, has_c, d_tma;
  float alpha, beta;
  uint16_t* D;  // the output of this thread's row block's matrix
  long long ldd;
  const CUtensorMap* tmD;
  int b;        // that matrix's index in its group
  int nb, kb;   // rows per block (128 / pack) and this thread's block (rows kb*nb .. +nb-1)
  int rl;       // this thread's row within its block
  bool valid;   // the block holds a matrix (the last job of a group may have fewer)
  bool badrow;  // the block's matrix is not finite: its X rows are kept at zero
};

// two 16-bit values of one word (the first in the low half) as fp32, and back (nearest even)
template <bool F16>
__device__ __forceinline__ float2 unpack2(uint32_t w) {
  if constexpr (F16) return __half22float2(*reinterpret_cast<const __half2*>(&w));
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));  // exact
}
template <bool F16>
__device__ __forceinline__ uint32_t pack2(float2 y) {
  if constexpr (F16) {
    const __half2 h = __float22half2_rn(y);
    return *reinterpret_cast<const uint32_t*>(&h);
  } else {
    const __nv_bfloat162 h = __float22bfloat162_rn(y);
    return *reinterpret_cast<const uint32_t*>(&h);
  }
}

// n x n products, one form per epilogue kind: E_SCALE y = k acc; E_POLY y = p1 acc + p0 C
// (and Q = y + p2 I when qinit); E_AXPY y = acc + p0 C. The addend chunks are read before
// anything is stored: C may be the output buffer itself (the in-place updates), and a load
// placed after a store to it could not start before it.
template <bool F16, int EPI>
__device__ __forceinline__ void nn_chunks(const Ctx& x, const Op o, int g, const float (&v)[32], float k, bool keep) {
  const int r = x.r;
  const int pb = (g >> 1) * PANEL_BYTES, jb = 4 * (g & 1);
  uint8_t* __restrict__ dp = x.sm + buf_off(o.d) + pb;
  const uint8_t* __restrict__ cp = x.sm + buf_off(o.c) + pb;
  uint8_t* __restrict__ qp = x.sm + OFF_Q + pb;
  uint4 cw[4];
  if constexpr (EPI != E_SCALE) {
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) cw[jj] = *reinterpret_cast<const uint4*>(cp + chunk_off(r, jb + jj));
  }
  const float2 k2 = make_float2(k, k), p0 = make_float2(o.p0, o.p0), p1 = make_float2(o.p1, o.p1);
  const bool qinit = EPI == E_POLY && (o.flags & F_QINIT) != 0;
#pragma unroll
  for (int jj = 0; jj < 4; ++jj) {
    const uint32_t cu[4] = {cw[jj].x, cw[jj].y, cw[jj].z, cw[jj].w};
    float2 y[4];
    uint32_t pk[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 a = make_float2(v[8 * jj + 2 * i], v[8 * jj + 2 * i + 1]);
      if constexpr (EPI == E_SCALE)
        y[i] = __fmul2_rn(k2, a);
      else if constexpr (EPI == E_POLY)
        y[i] = __ffma2_rn(p0, unpack2<F16>(cu[i]), __fmul2_rn(p1, a));
      else
        y[i] = __ffma2_rn(p0, unpack2<F16>(cu[i]), a);
      // packed chains: entries outside the diagonal blocks are exact zeros (selected, so that
      // a non-finite block cannot leak into the others)
      pk[i] = keep ? pack2<F16>(y[i]) : 0u;
    }
    const uint32_t off = chunk_off(r, jb + jj);
    *reinterpret_cast<uint4*>(dp + off) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
    if (qinit) *reinterpret_cast<uint4*>(qp + off) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
  }
  // Q = Z + a I: the diagonal entry (r, r) gets the fp32 value of Z plus a, rounded once
  // (Dion3 appendix B.2.3: adding a_t I to an already rounded Z would lose a_t's low bits);
  // rows at and beyond n (of the row's block) stay zero. Column r is local column lane of group r / 32, i.e. of
  // this group in the warps of lane quarter g (a warp-uniform test).
  if (qinit && g == (r >> 5)) {
    float ad = 0.f;
#pragma unroll
    for (int k2i = 0; k2i < 32; ++k2i)
      if (k2i == x.lane) ad = v[k2i];
    const uint32_t doff = (uint32_t)(r * 128 + (((jb + (x.lane >> 3)) ^ (r & 7)) << 4) + (x.lane & 7) * 2);
    const float zd = fmaf(o.p0, h16_to_f(*reinterpret_cast<const uint16_t*>(cp + doff), F16), o.p1 * ad);
    if (x.rl < x.n) *reinterpret_cast<uint16_t*>(qp + doff) = f_to_h16(zd + o.p2, F16);
  }
}

// All of this warp's 32-column groups of an n x n product (G = g, g + NG, ...). sc scales
// the accumulator of E_SCALE (s^2 for the Gram product of the user's X, else 1). (Both
// groups' TMEM loads in flight together spill registers at this kernel's budget.)
template <bool F16>
__device__ __forceinline__ void epi_nn(const Ctx& x, const Op o, float sc) {
#pragma unroll 1
  for (int G = x.g; G < 4; G += NG) {
    float v[32];
    load_acc32(x.trow, 128 * o.slot + 32 * G, v);
    const bool keep = (32 * G) / x.nb == x.kb;  // the group lies in this row's block
    if (o.epi == E_SCALE)
      nn_chunks<F16, E_SCALE>(x, o, G, v, sc, keep);
    else if (o.epi == E_POLY)
      nn_chunks<F16, E_POLY>(x, o, G, v, 1.f, keep);
    else
      nn_chunks<F16, E_AXPY>(x, o, G, v, 1.f, keep);
  }
}

// One 16-byte-aligned group of 4 output values: D = k y + beta D, non-finite results noted.
// vec: all 4 inside the matrix (else element by element, up to lim).
__device__ __forceinline__ bool out4(const Ctx& x, uint16_t* dst, const float4 y, float k, bool vec, int lim) {
  const int df = x.d_f16;
  const float2 k2 = make_float2(k, k), b2 = make_float2(x.beta, x.beta);
  float2 o0 = __fmul2_rn(k2, make_float2(y.x, y.y)), o1 = __fmul2_rn(k2, make_float2(y.z, y.w));
  bool bad = false;
  if (vec) {
    if (x.has_c) {
      const uint2 c = *reinterpret_cast<const uint2*>(dst);
      o0 = __ffma2_rn(b2, df ? unpack2<true>(c.x) : unpack2<false>(c.x), o0);
      o1 = __ffma2_rn(b2, df ? unpack2<true>(c.y) : unpack2<false>(c.y), o1);
    }
    bad = !(isfinite(o0.x) && isfinite(o0.y) && isfinite(o1.x) && isfinite(o1.y));
    *reinterpret_cast<uint2*>(dst) =
        df ? make_uint2(pack2<true>(o0), pack2<true>(o1)) : make_uint2(pack2<false>(o0), pack2<false>(o1));
  } else {
    const float ov[4] = {o0.x, o0.y, o1.x, o1.y};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      if (i >= lim) break;
      float t = ov[i];
      if (x.has_c) t = fmaf(x.beta, h16_to_f(dst[i], df), t);
      bad |= !isfinite(t);
      dst[i] = f_to_h16(t, df);
    }
  }
  return bad;
}

// A X products (n x m in TMEM columns 0 .. mp-1): this warp takes the 32-column groups
// G = g, g + 4, ... of its 32 rows. X <- Q X (E_XSET) and X <- a X + B X (E_XAXPY) write
// the region back in place (the products that read it have completed). The result (E_OUT)
// goes through a per-warp fp32 staging block (32 x 32) in the dead R and Z buffers, so that
// global memory sees row segments: 8 lanes per 32-column segment of a row of D, or for a
// transposed D (a tall matrix) 8 lanes per 32-row segment of one of its rows.
template <bool F16>
__device__ __forceinline__ bool epi_ax(const Ctx& x, const Op o, float s, int& nblk) {
  const int r = x.r, lane = x.lane;
  const float su = (o.flags & F_USER) ? s : 1.f;
  const bool out = o.epi == E_OUT;
  const bool rdx = o.epi == E_XAXPY || (o.flags & F_ADDX);
  const float2 p0 = make_float2(o.p0, o.p0), su2 = make_float2(su, su);
  const float kout = x.alpha * su;  // E_OUT: D = alpha su (acc [+ p0 X]) + beta D
  bool bad = false;
  uint8_t* __restrict__ stg = x.sm + OFF_R + x.ew * 4096;  // EPI_WARPS x 4 KiB <= R and Z
  // the op's 32-column groups [g0, g1): all, or one half, whose columns from ax_split(mp) lie
  // in TMEM from column 256 (tshift)
  const int gs = ax_split(x.mp) / 32;
  const int g0 = o.half == 1 ? gs : 0, g1 = o.half == 0 ? gs : x.mp / 32;
  const int tshift = o.half == 1 ? 256 - 32 * gs : 0;
  for (int G = g0 + x.g; G < g1; G += NG) {
    uint8_t* __restrict__ xp = x.sm + (G >> 1) * PANEL_BYTES;
    const int jb = 4 * (G & 1);
    uint4 cw[4];
    if (rdx) {
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) cw[jj] = *reinterpret_cast<const uint4*>(xp + chunk_off(r, jb + jj));
    }
    float v[32];
    load_acc32(x.trow, 32 * G + tshift, v);
    if (rdx) {
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) {
        const uint32_t cu[4] = {cw[jj].x, cw[jj].y, cw[jj].z, cw[jj].w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float2 t = __ffma2_rn(p0, unpack2<F16>(cu[i]), make_float2(v[8 * jj + 2 * i], v[8 * jj + 2 * i + 1]));
          v[8 * jj + 2 * i] = t.x;
          v[8 * jj + 2 * i + 1] = t.y;
        }
      }
    }
    if (!out) {
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) {
        uint32_t pk[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
          pk[i] = x.badrow ? 0u : pack2<F16>(__fmul2_rn(su2, make_float2(v[8 * jj + 2 * i], v[8 * jj + 2 * i + 1])));
        *reinterpret_cast<uint4*>(xp + chunk_off(r, jb + jj)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
      }
      continue;
    }
    // this warp's 32 rows lie in one block: rows row_q .. row_q + 31 of its matrix
    const int col_g = 32 * G, row_q = (r & ~31) % x.nb;
    if (x.badrow) {
      // a packed block whose input was not finite: its result is marked not finite (its
      // zeroed rows would otherwise give finite zeros after a restart)
#pragma unroll
      for (int i = 0; i < 32; ++i) v[i] = __int_as_float(0x7fc00000);
    }
    if (x.d_tma) {
      // D = alpha su acc, rounded once, staged as this warp's 32 x 32 block of 16-bit values
      // (64-byte rows, chunk c of row i at c ^ ((i / 2) mod 4): the TMA 64-byte swizzle) in one
      // of four 2 KiB buffers, and written by one TMA store (rows and columns outside D are
      // dropped by the copy itself)
      uint8_t* blk = x.sm + OFF_R + (4 * x.ew + (nblk & 3)) * 2048;
      if (lane == 0 && nblk >= 4) bulk_wait_read<3>();  // the store of four groups ago has read it
      __syncwarp();
      const float2 k2 = make_float2(kout, kout);
      float2 z = make_float2(0.f, 0.f);
      if (!x.d_trans) {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t pk[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float2 t = __fmul2_rn(k2, make_float2(v[8 * c + 2 * i], v[8 * c + 2 * i + 1]));
            z = __ffma2_rn(t, make_float2(0.f, 0.f), z);  // NaN once any value is not finite
            pk[i] = x.d_f16 ? pack2<true>(t) : pack2<false>(t);
          }
          *reinterpret_cast<uint4*>(blk + lane * 64 + ((c ^ ((lane >> 1) & 3)) << 4)) =
              make_uint4(pk[0], pk[1], pk[2], pk[3]);
        }
      } else {
        // transposed: row c of the block holds column c of O (the 32 values of this warp's rows)
#pragma unroll
        for (int c = 0; c < 32; c += 2) {
          const float2 t = __fmul2_rn(k2, make_float2(v[c], v[c + 1]));
          z = __ffma2_rn(t, make_float2(0.f, 0.f), z);
          const uint32_t pk = x.d_f16 ? pack2<true>(t) : pack2<false>(t);
          const uint32_t o0 = (uint32_t)(lane & 7) * 2 + ((uint32_t)((lane >> 3) ^ ((c >> 1) & 3)) << 4);
          const uint32_t o1 = (uint32_t)(lane & 7) * 2 + ((uint32_t)((lane >> 3) ^ (((c + 1) >> 1) & 3)) << 4);
          *reinterpret_cast<uint16_t*>(blk + c * 64 + o0) = (uint16_t)(pk & 0xFFFFu);
          *reinterpret_cast<uint16_t*>(blk + (c + 1) * 64 + o1) = (uint16_t)(pk >> 16);
        }
      }
      bad |= !(z.x == 0.f && z.y == 0.f) && x.rl < x.n && x.valid;
      fence_proxy_async_smem();
      __syncwarp();
      // (blocks wholly outside D, or of a job's missing matrices, are not stored)
      if (lane == 0 && x.valid && row_q < x.n && col_g < x.m) {
        if (!x.d_trans)
          tma_store_3d(x.tmD, blk, col_g, row_q, x.b);
        else
          tma_store_3d(x.tmD, blk, row_q, col_g, x.b);
      }
      if (lane == 0) bulk_commit();
      ++nblk;
      continue;
    }
    __syncwarp();  // the previous group's staging reads are done
    if (!x.d_trans) {
      // staging: row = lane (128 bytes), 16-byte chunk c at position c ^ (lane mod 8)
#pragma unroll
      for (int c = 0; c < 8; ++c)
        *reinterpret_cast<float4*>(stg + lane * 128 + ((c ^ (lane & 7)) << 4)) =
            make_float4(v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
      __syncwarp();
#pragma unroll 2
      for (int k = 0; k < 8; ++k) {
        const int rl = 4 * k + (lane >> 3), c = lane & 7;
        const int row = row_q + rl, col = col_g + 4 * c;
        const float4 y = *reinterpret_cast<const float4*>(stg + rl * 128 + ((c ^ (rl & 7)) << 4));
        if (x.valid && row < x.n && col < x.m)
          bad |= out4(x, x.D + (long long)row * x.ldd + col, y, kout, col + 4 <= x.m, x.m - col);
      }
    } else {
      // staging transposed: word (column c, lane) at c * 32 + lane
#pragma unroll
      for (int c = 0; c < 32; ++c) reinterpret_cast<float*>(stg)[c * 32 + lane] = v[c];
      __syncwarp();
#pragma unroll 2
      for (int k = 0; k < 8; ++k) {
        const int cl = 4 * k + (lane >> 3), gg = lane & 7;
        const int col = col_g + cl, row = row_q + 4 * gg;
        const float4 y = *reinterpret_cast<const float4*>(stg + cl * 128 + gg * 16);
        if (col < x.m && row < x.n)
          bad |= out4(x, x.D + (long long)col * x.ldd + row, y, kout, row + 4 <= x.n, x.n - row);
      }
    }
  }
  return bad;
}

// ------------------------------------------------------------------------------------
// the kernel: persistent CTAs, matrix b = blockIdx.x + i * gridDim.x

__global__ void __launch_bounds__(NUM_THREADS, 1) chain_kernel(const __grid_constant__ Params P) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(sm);
  uint64_t* bar_x = reinterpret_cast<uint64_t*>(sm + OFF_BAR);  // X landed (TMA transaction count)
  uint64_t* bar_acc = bar_x + 1;                                 // [op] its products completed
  uint64_t* bar_epi = bar_acc + MAX_OPS;                         // [op] its epilogue completed (8 warps)
  uint64_t* bar_norm = bar_epi + MAX_OPS;                        // norm partials written (8 warps)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_norm + 1);
  int* abort_word = reinterpret_cast<int*>(tmem_slot + 1);
  float* part = reinterpret_cast<float*>(tmem_slot + 2);         // [2][EPI_WARPS]
  volatile int* abortv = abort_word;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nops = P.nops;

  if (threadIdx.x == 0) {
    mbar_init(bar_x, 1);
    mbar_init(bar_norm, EPI_WARPS);
    for (int i = 0; i < nops; ++i) {
      mbar_init(&bar_acc[i], 1);
      mbar_init(&bar_epi[i], EPI_WARPS);
    }
    *abortv = 0;
    mbar_fence_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ---- X loads
    if (lane == 0) {
      int it = 0;
      bool issued = false;
      uint32_t ipar = 0;
      for (int i = blockIdx.x; i < P.total; i += gridDim.x, ++it) {
        const Group& gr = P.grp[group_of(P, i)];
        const int b = (i - gr.first) * gr.pack, mp = gr.mp, nb = gr.nb;
        const uint32_t xbytes = (uint32_t)(mp * 256);
        if (it > 0) {
          // the region is free once the last product (and, when its epilogue reads X, that
          // epilogue) of the previous matrix is done
          uint64_t* wb = P.ops[nops - 1].flags & F_ADDX ? &bar_epi[nops - 1] : &bar_acc[nops - 1];
          if (!mbar_wait(wb, (uint32_t)((it - 1) & 1), abortv, P.status)) break;
        }
        mbar_arrive_expect_tx(bar_x, xbytes);
        if (!gr.xt) {
          // the job's matrices b .. b + pack - 1 in row blocks of nb rows (a matrix index past
          // the group's last reads as zeros)
          for (int p = 0; p < mp / 64; ++p)
            for (int k = 0; k < gr.pack; ++k)
              tma_load_3d(sm + p * PANEL_BYTES + k * nb * 128, &gr.tmX, bar_x, 64 * p, 0, b + k);
        } else {
          for (int ib = 0; ib < 2; ++ib)
            for (int kb = 0; kb < mp / 64; ++kb)
              tma_load_3d(sm + ib * (mp * 128) + kb * 8192, &gr.tmX, bar_x, 64 * ib, 64 * kb, b);
        }
        issued = true;
        ipar = (uint32_t)(it & 1);
      }
      // no copy may still be writing shared memory when the CTA exits
      if (issued) {
        volatile int never = 0;
        mbar_wait(bar_x, ipar, &never, nullptr, 1000000000ull);
      }
    }
  } else if (warp == 1) {
    // ---- MMA issue
    if (lane == 0) {
      const int ab = P.ab_f16;
      int it = 0, last = -1;
      uint32_t last_par = 0;
      bool ok = true;
      for (int mi = blockIdx.x; ok && mi < P.total; mi += gridDim.x, ++it) {
        const uint32_t par = (uint32_t)(it & 1);
        const Group& gr = P.grp[group_of(P, mi)];
        const int mp = gr.mp;
        const bool xt_in = gr.xt != 0;
        for (int i = 0; i < nops; ++i) {
          const Op o = P.ops[i];
          if (i == 0) {
            // the previous matrix's last user of accumulator 0 has read it (later epilogues of
            // that matrix come before this one's in the epilogue warps' order); X has landed
            if (it > 0 && !(ok = mbar_wait(&bar_epi[P.op0_prev], par ^ 1u, abortv, P.status))) break;
            if (!(ok = mbar_wait(bar_x, par, abortv, P.status))) break;
          }
          if (o.dep >= 0 && !(ok = mbar_wait(&bar_epi[o.dep], par, abortv, P.status))) break;
          tc_fence_after();
          issue_op(o, mp, ab, xt_in, sbase, tmem);
          umma_commit(&bar_acc[i]);
          last = i;
          last_par = par;
        }
      }
      // the tensor memory is released only after the last issued products completed
      if (last >= 0) {
        volatile int never = 0;
        mbar_wait(&bar_acc[last], last_par, &never, nullptr, 1000000000ull);
      }
    }
  } else {
    // ---- epilogue
    const int ew = warp - FIRST_EPI_WARP;
    const int q = warp & 3;  // the TMEM lane quarter this warp may access
    const int g = ew >> 2;   // its first 32-column group (then every NG-th)
    const int r = 32 * q + lane;
    Ctx cx;
    cx.sm = sm;
    cx.trow = tmem + ((uint32_t)(32 * q) << 16);
    cx.r = r;
    cx.g = g;
    cx.ew = ew;
    cx.lane = lane;
    const bool f16 = P.ab_f16 != 0;
    int nblk = 0;  // TMA-stored result blocks of this warp
    const int norm_mode = P.norm_mode;
    const float eps = P.eps;
    // every wait of a warp is combined over its lanes, so that a timeout seen by one lane
    // takes the whole warp out of the loop together (the TMEM loads are warp-collective)
    int it = 0;
    bool ok = true, bad = false;
    for (int mi = blockIdx.x; ok && mi < P.total; mi += gridDim.x, ++it) {
      const uint32_t par = (uint32_t)(it & 1);
      const Group& gr = P.grp[group_of(P, mi)];
      const int pack = gr.pack, nb = gr.nb;
      cx.nb = nb;
      cx.kb = r / nb;
      cx.rl = r - cx.kb * nb;
      const int b = (mi - gr.first) * pack + cx.kb;  // this row block's matrix
      cx.valid = b < gr.count;
      cx.badrow = false;
      cx.n = gr.n;
      cx.m = gr.m;
      cx.mp = gr.mp;
      cx.d_f16 = gr.d_f16;
      cx.d_trans = gr.d_trans;
      cx.has_c = gr.has_c;
      cx.alpha = gr.alpha;
      cx.beta = gr.beta;
      cx.ldd = gr.ldd;
      cx.d_tma = gr.d_tma;
      cx.tmD = &gr.tmD;
      cx.D = static_cast<uint16_t*>(gr.D) + (long long)(cx.valid ? b : 0) * gr.sd;
      cx.b = b;
      float s = 1.f;
      if (norm_mode == 1 && cx.valid) s = gr.inv[b];
      // X has landed (the epilogues of X <- a X + B X and of the standard-NS result read it)
      if (!(ok = __all_sync(0xffffffffu, mbar_wait(bar_x, par, abortv, P.status)))) break;
      for (int i = 0; i < nops; ++i) {
        const Op o = P.ops[i];
        if (!(ok = __all_sync(0xffffffffu, mbar_wait(&bar_acc[i], par, abortv, P.status)))) break;
        tc_fence_after();
        if (o.kind == K_AX) {
          bad |= f16 ? epi_ax<true>(cx, o, s, nblk) : epi_ax<false>(cx, o, s, nblk);
          // the staging blocks lie in the R and Z buffers, which the next epilogues rewrite
          // (a first half is followed by the second, which stages in the same blocks in turn)
          if (o.epi == E_OUT && cx.d_tma && o.half != 0) {
            if (lane == 0) bulk_wait_read<0>();
            __syncwarp();
          }
        } else {
          if (i == 0) {
            // ||X||_F^2 = trace(X X^T): the diagonal of this accumulator (row r = 32 q + lane,
            // column r: local column lane of group q), summed per row block (one matrix each)
            // in a fixed order; a block whose sum is not finite has its X rows zeroed, so that
            // the products of a packed chain keep it from the other blocks. The exchange is
            // also the point from which every warp has finished the previous matrix (its
            // result staging in R and Z, read by its stores), before any warp writes R.
            const bool need = norm_mode == 2 || pack > 1;
            float d = 0.f;
            if (need && (q % NG) == g) {
              float v[32];
              load_acc32(cx.trow, 128 * o.slot + 32 * q, v);
#pragma unroll
              for (int k = 0; k < 32; ++k)
                if (k == lane) d = v[k];
            }
            d = warp_sum(d);
            if (lane == 0) part[par * EPI_WARPS + ew] = d;
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_norm);
            if (!(ok = __all_sync(0xffffffffu, mbar_wait(bar_norm, par, abortv, P.status)))) break;
            // fp32 throughout: the part's FP64 rate would make these few operations cost
            // microseconds
            float t = 0.f;
#pragma unroll
            for (int w = 0; w < EPI_WARPS; ++w)
              if ((32 * ((FIRST_EPI_WARP + w) & 3)) / nb == cx.kb) t += part[par * EPI_WARPS + w];
            if (norm_mode == 2 && (o.flags & F_USER)) s = 1.f / (sqrtf(t) + eps);
            if (pack > 1 && !isfinite(t)) {
              cx.badrow = true;
              for (int p = 0; p < cx.mp / 64; ++p)
#pragma unroll
                for (int j = 0; j < 8; ++j)
                  *reinterpret_cast<uint4*>(sm + p * PANEL_BYTES + chunk_off(r, j)) = make_uint4(0u, 0u, 0u, 0u);
            }
          }
          const float sc = (o.flags & F_USER) ? s * s : 1.f;
          if (f16)
            epi_nn<true>(cx, o, sc);
          else
            epi_nn<false>(cx, o, sc);
        }
        // shared-memory results visible to the MMAs (async proxy); TMEM reads ordered before
        // the arrival that frees the accumulator
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar_epi[i]);
      }
    }
    if (P.check_finite && __any_sync(0xffffffffu, bad) && lane == 0) set_status(P.status, GNS_DEVST_NONFINITE);
    if (lane == 0) bulk_wait_all();  // every result store has landed before the CTA exits
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace chain

// ------------------------------------------------------------------------------------
// host side

namespace {

using chain::Op;

// The op list of one matrix, with each op's dependency: the latest earlier op that wrote a
// buffer it reads or used one of its accumulators.
struct Builder {
  std::vector<Op> ops;
  int last_w[4] = {-1, -1, -1, -1};
  int last_slot[4] = {-1, -1, -1, -1};
  int next_slot = 0;
  int ax_slots = 4;
  void add(Op o, std::initializer_list<int> reads, std::initializer_list<int> writes) {
    int dep = -1;
    for (int bf : reads) dep = std::max(dep, last_w[bf]);
    int s0 = 0, ns = ax_slots;
    if (o.kind == chain::K_AX && o.half >= 0) {
      s0 = 2 * o.half;
      ns = 2;
    } else if (o.kind != chain::K_AX) {
      s0 = next_slot;
      ns = 1;
      next_slot = (next_slot + 1) & 3;
    }
    o.slot = (uint8_t)s0;
    for (int s = s0; s < s0 + ns; ++s) dep = std::max(dep, last_slot[s]);
    o.dep = (int16_t)dep;
    const int i = (int)ops.size();
    ops.push_back(o);
    for (int bf : writes) last_w[bf] = i;
    for (int s = s0; s < s0 + ns; ++s) last_slot[s] = i;
  }
};

Op make_op(uint8_t kind, uint8_t epi) {
  Op o;
  std::memset(&o, 0, sizeof(o));
  o.kind = kind;
  o.epi = epi;
  o.half = -1;
  return o;
}

// Dion3 Algorithm 3 (sec. 4.2), the step order of the batched path: R_0 = X X^T; per
// iteration Z = b R + c R^2 (Q = Z + a I while Q is the identity), RZ = R Z + a R,
// Q_t = Q Z + a Q, R_t = Z RZ + a RZ (R only where it is read again); a restart after
// iteration i forms X <- Q X, R <- X X^T, Q <- I; the result is Q_T X.
void build_gram(Builder& bd, const gns_ns_params& ns, bool user) {
  using namespace chain;
  bool xin = true;  // the region holds the input X (until the first restart overwrites it)
  auto fl = [&]() { return (uint8_t)((user ? F_USER : 0) | (xin ? F_XIN : 0)); };
  Op g = make_op(K_GRAM, E_SCALE);
  g.d = BUF_R;
  g.flags = fl();
  bd.add(g, {BUF_X}, {BUF_R});
  bool q_id = true;
  const int T = ns.T;
  for (int t = 1; t <= T; ++t) {
    const float a = ns.a[t - 1], b = ns.b[t - 1], c = ns.c[t - 1];
    if (t > 1 && ((ns.restart_mask >> (t - 1)) & 1u)) {
      Op x = make_op(K_AX, E_XSET);
      x.a = BUF_Q;
      x.flags = fl();
      bd.add(x, {BUF_Q, BUF_X}, {BUF_X});
      user = false;
      xin = false;
      Op r = make_op(K_GRAM, E_SCALE);
      r.d = BUF_R;
      bd.add(r, {BUF_X}, {BUF_R});
      q_id = true;
    }
    Op z = make_op(K_NN, E_POLY);
    z.a = z.b = z.c = BUF_R;
    z.d = BUF_Z;
    z.p0 = b;
    z.p1 = c;
    z.p2 = a;
    if (q_id) {
      z.flags = F_QINIT;
      bd.add(z, {BUF_R}, {BUF_Z, BUF_Q});
    } else {
      bd.add(z, {BUF_R}, {BUF_Z});
    }
    const bool r_needed = t < T && !((ns.restart_mask >> t) & 1u);
    if (r_needed) {  // RZ over R (on the critical path: issued before Q_t)
      Op o = make_op(K_NN, E_AXPY);
      o.a = BUF_R;
      o.b = BUF_Z;
      o.c = o.d = BUF_R;
      o.p0 = a;
      bd.add(o, {BUF_R, BUF_Z}, {BUF_R});
    }
    if (!q_id) {
      Op o = make_op(K_NN, E_AXPY);
      o.a = BUF_Q;
      o.b = BUF_Z;
      o.c = o.d = BUF_Q;
      o.p0 = a;
      bd.add(o, {BUF_Q, BUF_Z}, {BUF_Q});
    }
    if (r_needed) {  // R_t = Z RZ + a RZ, over RZ
      Op o = make_op(K_NN, E_AXPY);
      o.a = BUF_Z;
      o.b = BUF_R;
      o.c = o.d = BUF_R;
      o.p0 = a;
      bd.add(o, {BUF_Z, BUF_R}, {BUF_R});
    }
    q_id = false;
  }
  // the result in two column halves: the first half's epilogue runs under the second half's
  // products, and the next matrix's first product (accumulator 0) under the second half's
  // epilogue (the result writes nothing the products read)
  for (int h = 0; h < 2; ++h) {
    Op out = make_op(K_AX, E_OUT);
    out.a = BUF_Q;
    out.flags = fl();
    out.half = (int8_t)h;
    bd.add(out, {BUF_Q, BUF_X}, {});
  }
}

// Dion3 Algorithm 1 with the same products: A = X X^T, B = b A + c A^2, X <- a X + B X.
void build_std(Builder& bd, const gns_ns_params& ns, bool user) {
  using namespace chain;
  for (int t = 1; t <= ns.T; ++t) {
    const float a = ns.a[t - 1], b = ns.b[t - 1], c = ns.c[t - 1];
    const uint8_t uf = user ? F_USER : 0;
    Op g = make_op(K_GRAM, E_SCALE);
    g.d = BUF_R;
    g.flags = uf;
    bd.add(g, {BUF_X}, {BUF_R});
    Op z = make_op(K_NN, E_POLY);
    z.a = z.b = z.c = BUF_R;
    z.d = BUF_Z;
    z.p0 = b;
    z.p1 = c;
    bd.add(z, {BUF_R}, {BUF_Z});
    if (t < ns.T) {
      Op x = make_op(K_AX, E_XAXPY);
      x.a = BUF_Z;
      x.p0 = a;
      x.flags = uf;
      bd.add(x, {BUF_Z, BUF_X}, {BUF_X});
    } else {
      Op x = make_op(K_AX, E_OUT);
      x.a = BUF_Z;
      x.p0 = a;
      x.flags = (uint8_t)(uf | F_ADDX);
      bd.add(x, {BUF_Z, BUF_X}, {});
    }
    user = false;
  }
}

int count_ops(bool gram, const gns_ns_params& ns) {
  Builder bd;
  if (gram)
    build_gram(bd, ns, true);
  else
    build_std(bd, ns, true);
  return (int)bd.ops.size();
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn(std::string* err) {
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

}  // namespace

bool chain_supported(bool gram, gns_dtype dt, int64_t n, int64_t m, int xt, const gns_ns_params* ns) {
  const char* env = std::getenv("GNS_CHAIN_SMALL");  // read per call: tests compare both paths
  if ((env && env[0] == '0') || !ns) return false;
  if (dt != GNS_BF16 && dt != GNS_F16) return false;
  if (n < 1 || n > chain::NP || m < n || m > chain::MAXM) return false;
  if (!gram && xt) return false;
  return count_ops(gram, *ns) <= chain::MAX_OPS;
}

// Tensor map of a batch of 16-bit row-major matrices: dims {cols, rows, count} of the storage.
static bool encode16(CUtensorMap* map, const MatRef& mref, int64_t count, uint32_t box_cols, uint32_t box_rows,
                     int f16, CUtensorMapSwizzle swz, std::string* err) {
  auto fn = encode_fn(err);
  if (!fn) return false;
  int64_t st_b = (count > 1 ? mref.stride : mref.rows * mref.ld) * 2;
  st_b = std::max<int64_t>((st_b + 15) / 16 * 16, 16);
  cuuint64_t dims[3] = {(cuuint64_t)mref.cols, (cuuint64_t)mref.rows, (cuuint64_t)count};
  cuuint64_t strides[2] = {(cuuint64_t)(mref.ld * 2), (cuuint64_t)st_b};
  cuuint32_t box[3] = {box_cols, box_rows, 1u};
  cuuint32_t estr[3] = {1u, 1u, 1u};
  const CUresult r = fn(map, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, mref.ptr,
                        dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    *err = "cuTensorMapEncodeTiled failed (code " + std::to_string((int)r) + ")";
    return false;
  }
  return true;
}

int launch_chain(const ChainCall& c, std::string* err) {
  using namespace chain;
  if (c.groups.empty()) return GNS_OK;
  for (const ChainGroup& g : c.groups)
    if (!chain_supported(c.gram, c.dt, g.n, g.m, g.xt, c.ns) || (c.x_user && (g.inv == nullptr) != (c.groups[0].inv == nullptr))) {
      *err = "chain kernel: unsupported group";
      return GNS_ERR_UNSUPPORTED;
    }
  Builder bd;  // one op list for every group: X <- Q X and Q X take all four accumulators
  if (c.gram)
    build_gram(bd, *c.ns, c.x_user);
  else
    build_std(bd, *c.ns, c.x_user);

  static bool attr_set[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) dev = 0;
  if (!attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(chain_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) {
      *err = std::string("cudaFuncSetAttribute: ") + cudaGetErrorString(e);
      return GNS_ERR_CUDA;
    }
    attr_set[dev] = true;
  }

  // up to MAX_GROUPS groups per launch; the launch's matrices are the groups' matrices in order
  thread_local Params P;  // a few KB (tensor maps, op list): built per calling thread, copied at launch
  const int f16 = c.dt == GNS_F16;
  for (size_t g0 = 0; g0 < c.groups.size(); g0 += MAX_GROUPS) {
    std::memset(&P, 0, sizeof(P));
    P.nops = (int)bd.ops.size();
    for (int i = 0; i < P.nops; ++i) P.ops[i] = bd.ops[i];
    P.op0_prev = bd.last_slot[0];
    P.ab_f16 = f16;
    P.norm_mode = !c.x_user ? 0 : c.groups[0].inv ? 1 : 2;
    P.eps = c.eps;
    P.check_finite = c.check_finite;
    P.status = c.status;
    int64_t total = 0;
    const size_t g1 = std::min(c.groups.size(), g0 + MAX_GROUPS);
    for (size_t gi = g0; gi < g1; ++gi) {
      const ChainGroup& cg = c.groups[gi];
      Group& G = P.grp[P.ngroups++];
      // wide matrices of at most 64 (32) rows go two (four) to a 128-row chain, each in a
      // diagonal block of the iterates (GNS_CHAIN_PACK=0 turns this off)
      const char* penv = std::getenv("GNS_CHAIN_PACK");
      const bool pack_ok = !cg.xt && !(penv && penv[0] == '0');
      G.pack = pack_ok && cg.n <= 32 ? 4 : pack_ok && cg.n <= 64 ? 2 : 1;
      G.nb = NP / G.pack;
      G.first = (int)total;
      G.count = (int)cg.B;
      total += (cg.B + G.pack - 1) / G.pack;
      G.n = (int)cg.n;
      G.m = (int)cg.m;
      G.mp = (int)((cg.m + 63) / 64 * 64);
      G.xt = cg.xt;
      G.inv = cg.inv;
      G.D = cg.D.ptr;
      G.ldd = cg.D.ld;
      G.sd = cg.B > 1 ? cg.D.stride : 0;
      G.d_f16 = cg.d_f16;
      G.d_trans = cg.d_trans;
      G.has_c = cg.has_c;
      G.alpha = cg.alpha;
      G.beta = cg.beta;
      // X: rows of the n x m operand (box 64 columns x 128 rows), or for a tall matrix its
      // m x n storage (box 64 x 64); zero fill outside the matrix
      if (!encode16(&G.tmX, cg.x, cg.B, 64u, cg.xt ? 64u : (uint32_t)G.nb, f16, CU_TENSOR_MAP_SWIZZLE_128B, err))
        return GNS_ERR_CUDA;
      // the result, when no addend is read: 32 x 32 boxes of its storage
      G.d_tma = !cg.has_c;
      if (G.d_tma && !encode16(&G.tmD, cg.D, cg.B, 32u, 32u, cg.d_f16, CU_TENSOR_MAP_SWIZZLE_64B, err))
        return GNS_ERR_CUDA;
    }
    if (total > INT32_MAX) {
      *err = "chain kernel: too many matrices in one launch";
      return GNS_ERR_UNSUPPORTED;
    }
    P.total = (int)total;
    const int grid = (int)std::min<int64_t>(total, device_sm_count());
    profile_gemm_begin(c.stream);
    chain_kernel<<<grid, NUM_THREADS, SMEM_BYTES, static_cast<cudaStream_t>(c.stream)>>>(P);
    const cudaError_t e = cudaGetLastError();
    profile_gemm_end(c.stream);
    if (e != cudaSuccess) {
      *err = std::string("chain_kernel launch: ") + cudaGetErrorString(e);
      return GNS_ERR_CUDA;
    }
  }
  return GNS_OK;
}

}  // namespace gns
