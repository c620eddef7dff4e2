// Batched bf16 GEMM on the 5th-generation tensor cores (tcgen05 + TMEM + TMA), sm_103a.
//
// One persistent CTA per SM walks a list of 128 x 128 output tiles (all tiles of a
// rectangular product, or the upper-triangle tiles of a symmetric one: Dion3 sec. 5
// "Triangular Scheduler"). Warp roles:
//   warp 0    TMA producer: 64-wide K slices of A and B into a 4-stage shared-memory ring
//             (128-byte swizzle; K-major operands as one 128x64 box, MN-major ones as two
//             64x64 boxes), completion on per-stage mbarriers.
//   warp 1    TMEM allocator and MMA issuer: one thread issues tcgen05.mma (M=128, N=128,
//             K=16, bf16 in, fp32 accumulate) into one of two TMEM accumulators, so the
//             epilogue of tile i overlaps the main loop of tile i+1 (Dion3 appendix C.1).
//   warps 2-5 epilogue: tcgen05.ld of the accumulator (thread = tile row), alpha/beta
//             combination with the C tile staged in shared memory, store through shared
//             staging with coalesced global writes; symmetric tiles are also written
//             transposed to the mirrored position, diagonal tiles once (Dion3 sec. 5
//             "Writing to the Transposed Tile", appendix C.1).
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>
#include <vector>

#include "common.cuh"
#include "gemm.h"

namespace gns {

namespace tc {

constexpr int TM = 128;
constexpr int TN = 128;
constexpr int TK = 64;
constexpr int STAGES = 4;
constexpr int A_BYTES = TM * TK * 2;                 // 16 KiB
constexpr int STAGE_BYTES = (TM + TN) * TK * 2;      // 32 KiB
constexpr int SPITCH = TN + 8;                       // staging row pitch (elements)
constexpr int STAGING_BYTES = TM * SPITCH * 2;       // 34816
constexpr int NUM_THREADS = 192;
constexpr int MAX_PROB = 4;
constexpr int TMEM_COLS = 256;                       // two 128-column fp32 accumulators
constexpr int BAR_BYTES = 256;
constexpr int DIAG_BYTES = TM * 4;                   // fp32 diagonal of a tile (for D2)
constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + 2 * STAGING_BYTES + BAR_BYTES + DIAG_BYTES;

struct Problem {
  CUtensorMap tmA;
  CUtensorMap tmB;
  int a_mn, b_mn;
  int M, N;
  int kblocks;
  int tiles_m, tiles_n, sym;
  int tile_begin, tiles_per_mat;
  float alpha, beta, gamma;
  int alpha_pow, beta_pow;
  const float* scale;
  const bf16* C;
  long long ldc, sc;
  int c_trans;
  bf16* D;
  long long ldd, sd;
  int d_trans;
  bf16* D2;
  long long ld2, s2;
  int diag_limit;
  const int* row_map;
  long long rm_stride;
  int check_finite;
};

struct Params {
  Problem prob[MAX_PROB];
  int nprob;
  int total_tiles;
  int* status;
};

struct TileCoord {
  int p, b, tm, tn;
};

__device__ __forceinline__ TileCoord decode_tile(const Params& P, int tile) {
  TileCoord tc;
  int p = 0;
  while (p + 1 < P.nprob && tile >= P.prob[p + 1].tile_begin) ++p;
  const Problem& pr = P.prob[p];
  int t = tile - pr.tile_begin;
  tc.p = p;
  tc.b = t / pr.tiles_per_mat;
  t -= tc.b * pr.tiles_per_mat;
  if (pr.sym) {
    int i = 0;
    while (t >= pr.tiles_m - i) {
      t -= pr.tiles_m - i;
      ++i;
    }
    tc.tm = i;
    tc.tn = i + t;
  } else {
    tc.tm = t / pr.tiles_n;
    tc.tn = t - tc.tm * pr.tiles_n;
  }
  return tc;
}

__device__ __forceinline__ float powi(float s, int p) { return p == 0 ? 1.f : (p == 1 ? s : s * s); }

// Staging block S (128 x 128, pitch SPITCH) <-> global matrix G of batch entry b:
//   trans = 0: S[u][v] = G[pi(m0+u)][n0+v]   (valid when m0+u < M and n0+v < N)
//   trans = 1: S[u][v] = G[n0+u][pi(m0+v)]   (valid when n0+u < N and m0+v < M)
// pi(i) = row_map ? row_map[b*rms + i] : i. Out-of-range elements load as 0 and are not stored.
__device__ void coop_load(bf16* S, const bf16* G, long long ld, long long sb, int b, int trans, int m0, int n0,
                          int M, int N, const int* row_map, long long rms, int et) {
  const int ew = et >> 5, lane = et & 31;
  const bf16* Gb = G + (long long)b * sb;
  const int v0 = lane * 4;
  for (int u = ew; u < TM; u += 4) {
    uint2 pk = make_uint2(0u, 0u);
    bf16* pv = reinterpret_cast<bf16*>(&pk);
    if (!trans) {
      const int gi = m0 + u;
      const int gj = n0 + v0;
      if (gi < M) {
        const long long ro = (long long)(row_map ? row_map[(long long)b * rms + gi] : gi) * ld;
        if (gj + 3 < N) {
          pk = *reinterpret_cast<const uint2*>(Gb + ro + gj);
        } else {
          for (int e = 0; e < 4; ++e)
            if (gj + e < N) pv[e] = Gb[ro + gj + e];
        }
      }
    } else {
      const int gj = n0 + u;
      const int gi = m0 + v0;
      if (gj < N) {
        const long long ro = (long long)gj * ld;
        if (!row_map && gi + 3 < M) {
          pk = *reinterpret_cast<const uint2*>(Gb + ro + gi);
        } else {
          for (int e = 0; e < 4; ++e)
            if (gi + e < M) pv[e] = Gb[ro + (row_map ? row_map[(long long)b * rms + gi + e] : gi + e)];
        }
      }
    }
    *reinterpret_cast<uint2*>(S + u * SPITCH + v0) = pk;
  }
}

// Inverse of coop_load; also writes D2 = D + gamma I when D2 is set (same row mapping as
// D): off the diagonal D2 takes the stored value, on the global diagonal (gi == gj <
// diag_limit) it takes dg[u], the fp32 diagonal plus gamma rounded once (appendix B.2.3:
// adding a_t I to an already rounded Z loses a_t's precision).
__device__ void coop_store(const bf16* S, bf16* G, long long ld, long long sb, bf16* G2, long long ld2,
                           long long sb2, const float* dg, int diag_limit, int b, int trans, int m0, int n0, int M,
                           int N, const int* row_map, long long rms, int et) {
  const int ew = et >> 5, lane = et & 31;
  bf16* Gb = G + (long long)b * sb;
  bf16* G2b = G2 ? G2 + (long long)b * sb2 : nullptr;
  const int v0 = lane * 4;
  for (int u = ew; u < TM; u += 4) {
    const uint2 pk = *reinterpret_cast<const uint2*>(S + u * SPITCH + v0);
    const bf16* pv = reinterpret_cast<const bf16*>(&pk);
    if (!trans) {
      const int gi = m0 + u;
      const int gj = n0 + v0;
      if (gi >= M) continue;
      const int pi = row_map ? row_map[(long long)b * rms + gi] : gi;
      const long long ro = (long long)pi * ld;
      if (gj + 3 < N) {
        *reinterpret_cast<uint2*>(Gb + ro + gj) = pk;
      } else {
        for (int e = 0; e < 4; ++e)
          if (gj + e < N) Gb[ro + gj + e] = pv[e];
      }
      if (G2b) {
        const long long ro2 = (long long)pi * ld2;
        uint2 q = pk;
        bf16* qv = reinterpret_cast<bf16*>(&q);
        for (int e = 0; e < 4; ++e)
          if (gi == gj + e && gi < diag_limit) qv[e] = f_to_bf16(dg[u]);
        if (gj + 3 < N) {
          *reinterpret_cast<uint2*>(G2b + ro2 + gj) = q;
        } else {
          for (int e = 0; e < 4; ++e)
            if (gj + e < N) G2b[ro2 + gj + e] = qv[e];
        }
      }
    } else {
      const int gj = n0 + u;
      const int gi = m0 + v0;
      if (gj >= N) continue;
      const long long ro = (long long)gj * ld;
      if (!row_map && gi + 3 < M) {
        *reinterpret_cast<uint2*>(Gb + ro + gi) = pk;
      } else {
        for (int e = 0; e < 4; ++e)
          if (gi + e < M) Gb[ro + (row_map ? row_map[(long long)b * rms + gi + e] : gi + e)] = pv[e];
      }
    }
  }
}

__global__ void __launch_bounds__(NUM_THREADS, 1) gemm_kernel(const __grid_constant__ Params P) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* stages = smem;
  bf16* S0 = reinterpret_cast<bf16*>(smem + STAGES * STAGE_BYTES);
  bf16* S1 = S0 + TM * SPITCH;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES + 2 * STAGING_BYTES);
  uint64_t* full = bars;
  uint64_t* empty = bars + STAGES;
  uint64_t* tfull = bars + 2 * STAGES;
  uint64_t* tempty = tfull + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tempty + 2);
  float* diag = reinterpret_cast<float*>(smem + STAGES * STAGE_BYTES + 2 * STAGING_BYTES + BAR_BYTES);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* epi_flag = abort_flag + 1;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 128);
    }
    *abort_flag = 0;
    *epi_flag = 1;
    mbar_fence_init();
  }
  if (warp == 0 && lane == 0) {
    for (int p = 0; p < P.nprob; ++p) {
      tma_prefetch_desc(&P.prob[p].tmA);
      tma_prefetch_desc(&P.prob[p].tmB);
    }
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer ----------------
      int s = 0;
      uint32_t ph = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < P.total_tiles; tile += gridDim.x) {
        const TileCoord c = decode_tile(P, tile);
        const Problem& pr = P.prob[c.p];
        const int m0 = c.tm * TM, n0 = c.tn * TN;
        for (int kb = 0; kb < pr.kblocks; ++kb) {
          if (!mbar_wait(&empty[s], ph ^ 1u, abort_flag, P.status)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full[s], STAGE_BYTES);
          uint8_t* sa = stages + s * STAGE_BYTES;
          uint8_t* sb = sa + A_BYTES;
          const int k0 = kb * TK;
          if (!pr.a_mn) {
            tma_load_3d(sa, &pr.tmA, &full[s], k0, m0, c.b);
          } else {
            tma_load_3d(sa, &pr.tmA, &full[s], m0, k0, c.b);
            tma_load_3d(sa + 8192, &pr.tmA, &full[s], m0 + 64, k0, c.b);
          }
          if (!pr.b_mn) {
            tma_load_3d(sb, &pr.tmB, &full[s], k0, n0, c.b);
          } else {
            tma_load_3d(sb, &pr.tmB, &full[s], n0, k0, c.b);
            tma_load_3d(sb + 8192, &pr.tmB, &full[s], n0 + 64, k0, c.b);
          }
          if (++s == STAGES) {
            s = 0;
            ph ^= 1u;
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer ----------------
      int s = 0;
      uint32_t ph = 0;
      bool ok = true;
      int local = 0;
      for (int tile = blockIdx.x; ok && tile < P.total_tiles; tile += gridDim.x, ++local) {
        const TileCoord c = decode_tile(P, tile);
        const Problem& pr = P.prob[c.p];
        const int acc = local & 1;
        const uint32_t aph = (local >> 1) & 1;
        if (!mbar_wait(&tempty[acc], aph ^ 1u, abort_flag, P.status)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * TN;
        const uint32_t idesc = idesc_bf16_f32(TM, TN, pr.a_mn, pr.b_mn);
        for (int kb = 0; kb < pr.kblocks; ++kb) {
          if (!mbar_wait(&full[s], ph, abort_flag, P.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(stages + s * STAGE_BYTES);
          const uint32_t sb = sa + A_BYTES;
#pragma unroll
          for (int kk = 0; kk < TK / 16; ++kk) {
            const uint64_t ad = pr.a_mn ? sdesc_sw128(sa + kk * 2048, 8192, 1024) : sdesc_sw128(sa + kk * 32, 16, 1024);
            const uint64_t bd = pr.b_mn ? sdesc_sw128(sb + kk * 2048, 8192, 1024) : sdesc_sw128(sb + kk * 32, 16, 1024);
            umma_bf16(d_tmem, ad, bd, idesc, (kb | kk) != 0 ? 1u : 0u);
          }
          umma_commit(&empty[s]);
          if (++s == STAGES) {
            s = 0;
            ph ^= 1u;
          }
        }
        if (ok) umma_commit(&tfull[acc]);
      }
    }
  } else {
    // ---------------- epilogue (warps 2..5) ----------------
    const int et = threadIdx.x - 64;
    const int quarter = warp & 3;  // TMEM lanes this warp may read
    const int r = quarter * 32 + lane;
    int local = 0;
    for (int tile = blockIdx.x; tile < P.total_tiles; tile += gridDim.x, ++local) {
      const TileCoord c = decode_tile(P, tile);
      const Problem& pr = P.prob[c.p];
      const int acc = local & 1;
      const uint32_t aph = (local >> 1) & 1;
      float alpha = pr.alpha, beta = pr.beta;
      if (pr.scale) {
        const float sc = pr.scale[c.b];
        alpha *= powi(sc, pr.alpha_pow);
        beta *= powi(sc, pr.beta_pow);
      }
      const bool has_c = pr.C != nullptr && beta != 0.f;
      const bool mirror = pr.sym && c.tm != c.tn;
      const int m0 = c.tm * TM, n0 = c.tn * TN;
      if (has_c) coop_load(S0, pr.C, pr.ldc, pr.sc, c.b, pr.c_trans, m0, n0, pr.M, pr.N, pr.row_map, pr.rm_stride, et);
      if (et == 0) *epi_flag = mbar_wait(&tfull[acc], aph, abort_flag, P.status) ? 1 : 0;
      named_bar_sync(1, 128);
      if (!*epi_flag) break;
      tc_fence_after();
      const bool inplace = !has_c || (pr.c_trans == pr.d_trans);
      bf16* SD = inplace ? S0 : S1;
      const bool want_diag = pr.D2 != nullptr && c.tm == c.tn;
      float dv = 0.f;
      bool bad = false;
#pragma unroll 1
      for (int ch = 0; ch < TN / 32; ++ch) {
        uint32_t v[32];
        __syncwarp();  // tcgen05.ld is warp-aligned
        tmem_ld_32x32b_x32(tmem_base + acc * TN + ch * 32 + ((uint32_t)(quarter * 32) << 16), v);
        tmem_ld_wait();
        float o[32];
        if (has_c) {
          if (!pr.c_trans) {
            const uint4* src = reinterpret_cast<const uint4*>(S0 + r * SPITCH + ch * 32);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const uint4 w = src[q];
              const bf16* wv = reinterpret_cast<const bf16*>(&w);
#pragma unroll
              for (int e = 0; e < 8; ++e) o[q * 8 + e] = beta * bf16_to_f(wv[e]);
            }
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) o[j] = beta * bf16_to_f(S0[(ch * 32 + j) * SPITCH + r]);
          }
#pragma unroll
          for (int j = 0; j < 32; ++j) o[j] = fmaf(alpha, __uint_as_float(v[j]), o[j]);
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) o[j] = alpha * __uint_as_float(v[j]);
        }
        if (pr.check_finite) {
#pragma unroll
          for (int j = 0; j < 32; ++j) bad |= !isfinite(o[j]);
        }
        if (want_diag && (r >> 5) == ch) {
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (j == (r & 31)) dv = o[j];
        }
        if (!pr.d_trans) {
          uint4* dst = reinterpret_cast<uint4*>(SD + r * SPITCH + ch * 32);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint4 w;
            bf16* wv = reinterpret_cast<bf16*>(&w);
#pragma unroll
            for (int e = 0; e < 8; ++e) wv[e] = f_to_bf16(o[q * 8 + e]);
            dst[q] = w;
          }
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) SD[(ch * 32 + j) * SPITCH + r] = f_to_bf16(o[j]);
        }
        if (mirror) {
#pragma unroll
          for (int j = 0; j < 32; ++j) S1[(ch * 32 + j) * SPITCH + r] = f_to_bf16(o[j]);
        }
      }
      if (want_diag) diag[r] = dv + pr.gamma;
      tc_fence_before();
      mbar_arrive(&tempty[acc]);
      if (bad) set_status(P.status, GNS_DEVST_NONFINITE);
      named_bar_sync(1, 128);
      coop_store(SD, pr.D, pr.ldd, pr.sd, pr.D2, pr.ld2, pr.s2, diag, pr.diag_limit, c.b, pr.d_trans, m0, n0,
                 pr.M, pr.N, pr.row_map, pr.rm_stride, et);
      if (mirror)
        coop_store(S1, pr.D, pr.ldd, pr.sd, pr.D2, pr.ld2, pr.s2, diag, pr.diag_limit, c.b, 0, n0, m0, pr.N,
                   pr.M, nullptr, 0, et);
      named_bar_sync(1, 128);
    }
  }

  // lanes 1-31 of the producer and MMA warps wait here for lane 0 (aligned barrier below)
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
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

// 3-D bf16 tensor map over a batch of row-major matrices: dims {cols, rows, batch}.
static bool encode_map(CUtensorMap* map, const MatRef& m, int64_t batch, bool kmajor, std::string* err) {
  auto fn = get_encode_fn(err);
  if (!fn) return false;
  const int64_t ld_b = m.ld * 2;
  int64_t st_b = (batch > 1 ? m.stride : m.rows * m.ld) * 2;
  st_b = (st_b + 15) / 16 * 16;
  if (st_b == 0) st_b = 16;
  cuuint64_t dims[3] = {(cuuint64_t)m.cols, (cuuint64_t)m.rows, (cuuint64_t)batch};
  cuuint64_t strides[2] = {(cuuint64_t)ld_b, (cuuint64_t)st_b};
  cuuint32_t box[3] = {64u, kmajor ? 128u : 64u, 1u};
  cuuint32_t estr[3] = {1u, 1u, 1u};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, m.ptr, dims, strides, box, estr,
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

int gemm_launch_bf16(const GemmOp* ops, int nops, int32_t* dev_status, void* stream, std::string* err) {
  using namespace tc;
  if (nops < 1 || nops > MAX_PROB) {
    *err = "internal: bad number of grouped products";
    return GNS_ERR_INVALID;
  }
  static bool attr_set[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) {
      *err = std::string("cudaFuncSetAttribute: ") + cudaGetErrorString(e);
      return GNS_ERR_CUDA;
    }
    attr_set[dev] = true;
  }
  Params P;
  memset(&P, 0, sizeof(P));
  int tiles = 0;
  for (int i = 0; i < nops; ++i) {
    const GemmOp& o = ops[i];
    Problem& pr = P.prob[i];
    if (!encode_map(&pr.tmA, o.A, o.batch, !o.a_mn, err)) return GNS_ERR_CUDA;
    if (!encode_map(&pr.tmB, o.B, o.batch, !o.b_mn, err)) return GNS_ERR_CUDA;
    pr.a_mn = o.a_mn;
    pr.b_mn = o.b_mn;
    pr.M = (int)o.M;
    pr.N = (int)o.N;
    pr.kblocks = (int)((o.K + TK - 1) / TK);
    pr.tiles_m = (int)((o.M + TM - 1) / TM);
    pr.tiles_n = (int)((o.N + TN - 1) / TN);
    pr.sym = o.sym;
    pr.tiles_per_mat = o.sym ? pr.tiles_m * (pr.tiles_m + 1) / 2 : pr.tiles_m * pr.tiles_n;
    pr.tile_begin = tiles;
    tiles += pr.tiles_per_mat * (int)o.batch;
    pr.alpha = o.alpha;
    pr.beta = o.beta;
    pr.gamma = o.gamma;
    pr.alpha_pow = o.alpha_pow;
    pr.beta_pow = o.beta_pow;
    pr.scale = o.scale;
    pr.C = static_cast<const bf16*>(o.C.ptr);
    pr.ldc = o.C.ld;
    pr.sc = o.C.stride;
    pr.c_trans = o.c_trans;
    pr.D = static_cast<bf16*>(o.D.ptr);
    pr.ldd = o.D.ld;
    pr.sd = o.D.stride;
    pr.d_trans = o.d_trans;
    pr.D2 = static_cast<bf16*>(o.D2.ptr);
    pr.ld2 = o.D2.ld;
    pr.s2 = o.D2.stride;
    pr.diag_limit = (int)o.diag_limit;
    pr.row_map = o.row_map;
    pr.rm_stride = o.row_map_stride;
    pr.check_finite = o.check_finite;
  }
  P.nprob = nops;
  P.total_tiles = tiles;
  P.status = dev_status;
  if (tiles == 0) return GNS_OK;
  const int grid = std::min(tiles, device_sm_count());
  gemm_kernel<<<grid, NUM_THREADS, SMEM_BYTES, static_cast<cudaStream_t>(stream)>>>(P);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    *err = std::string("tcgen05 GEMM launch: ") + cudaGetErrorString(e);
    return GNS_ERR_CUDA;
  }
  return GNS_OK;
}

}  // namespace gns
