// Batched fp32 GEMM on the CUDA cores (FFMA): the validation path of libgns.
//
// Same operand/epilogue contract as the tensor-core kernel (gemm.h) but in fp32 end to
// end, so that the whole Gram Newton-Schulz sequence can be checked against the fp64
// oracle to 1e-4. 64 x 64 output tiles, 256 threads (4 x 4 outputs each), K slices of 16
// staged in shared memory; symmetric products compute upper-triangle tiles only and write
// off-diagonal tiles twice (direct and mirrored), diagonal tiles once.
#include <algorithm>

#include "common.cuh"
#include "gemm.h"

namespace gns {

namespace simt {

constexpr int T = 64;
constexpr int BK = 16;
constexpr int MAX_PROB = 4;

struct Problem {
  const float* A;
  long long lda, sa;
  int a_mn;
  const float* B;
  long long ldb, sb;
  int b_mn;
  int M, N, K;
  int am, ak, bn, bk;  // valid extents of A (rows i, depth k) and B (rows j, depth k)
  int tiles_m, tiles_n, sym, tile_begin, tiles_per_mat;
  float alpha, beta, gamma;
  int alpha_pow, beta_pow;
  const float* scale;
  const float* C;
  long long ldc, sc;
  int c_trans;
  float* D;
  long long ldd, sd;
  int d_trans;
  float* D2;
  long long ld2, s2;
  int diag_limit;
  const int* row_map;
  long long rms;
  int check_finite;
};

struct Params {
  Problem prob[MAX_PROB];
  int nprob;
  int total_tiles;
  int* status;
};

__device__ __forceinline__ float powi(float s, int p) { return p == 0 ? 1.f : (p == 1 ? s : s * s); }

__global__ void __launch_bounds__(256) gemm_kernel(const __grid_constant__ Params P) {
  __shared__ float As[BK][T + 4];
  __shared__ float Bs[BK][T + 4];
  __shared__ int bad_any;
  const int tid = threadIdx.x;
  for (int tile = blockIdx.x; tile < P.total_tiles; tile += gridDim.x) {
    int p = 0;
    while (p + 1 < P.nprob && tile >= P.prob[p + 1].tile_begin) ++p;
    const Problem& pr = P.prob[p];
    int t = tile - pr.tile_begin;
    const int b = t / pr.tiles_per_mat;
    t -= b * pr.tiles_per_mat;
    int tm, tn;
    if (pr.sym) {
      int i = 0;
      while (t >= pr.tiles_m - i) {
        t -= pr.tiles_m - i;
        ++i;
      }
      tm = i;
      tn = i + t;
    } else {
      tm = t / pr.tiles_n;
      tn = t - tm * pr.tiles_n;
    }
    const int m0 = tm * T, n0 = tn * T;
    const float* A = pr.A + (long long)b * pr.sa;
    const float* B = pr.B + (long long)b * pr.sb;
    const int tx = tid & 15, ty = tid >> 4;
    float acc[4][4] = {};
    if (tid == 0) bad_any = 0;
    for (int k0 = 0; k0 < pr.K; k0 += BK) {
      // 64 x 16 slices of A and B, 4 elements per thread each
      for (int e = tid; e < T * BK; e += 256) {
        int i, k;
        if (pr.a_mn) {
          k = e / T;
          i = e % T;
        } else {
          i = e / BK;
          k = e % BK;
        }
        const int gi = m0 + i, gk = k0 + k;
        float va = 0.f;
        if (gi < pr.am && gk < pr.ak) va = pr.a_mn ? A[(long long)gk * pr.lda + gi] : A[(long long)gi * pr.lda + gk];
        As[k][i] = va;
        int j, kb;
        if (pr.b_mn) {
          kb = e / T;
          j = e % T;
        } else {
          j = e / BK;
          kb = e % BK;
        }
        const int gj = n0 + j, gkb = k0 + kb;
        float vb = 0.f;
        if (gj < pr.bn && gkb < pr.bk) vb = pr.b_mn ? B[(long long)gkb * pr.ldb + gj] : B[(long long)gj * pr.ldb + gkb];
        Bs[kb][j] = vb;
      }
      __syncthreads();
#pragma unroll
      for (int k = 0; k < BK; ++k) {
        float a[4], bb[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          a[q] = As[k][ty * 4 + q];
          bb[q] = Bs[k][tx * 4 + q];
        }
#pragma unroll
        for (int q = 0; q < 4; ++q)
#pragma unroll
          for (int w = 0; w < 4; ++w) acc[q][w] = fmaf(a[q], bb[w], acc[q][w]);
      }
      __syncthreads();
    }
    float alpha = pr.alpha, beta = pr.beta;
    if (pr.scale) {
      alpha *= powi(pr.scale[b], pr.alpha_pow);
      beta *= powi(pr.scale[b], pr.beta_pow);
    }
    const bool has_c = pr.C && beta != 0.f;
    const bool mirror = pr.sym && tm != tn;
    bool bad = false;
    for (int q = 0; q < 4; ++q) {
      const int gi = m0 + ty * 4 + q;
      if (gi >= pr.M) continue;
      const int pi = pr.row_map ? pr.row_map[(long long)b * pr.rms + gi] : gi;
      for (int w = 0; w < 4; ++w) {
        const int gj = n0 + tx * 4 + w;
        if (gj >= pr.N) continue;
        float o = alpha * acc[q][w];
        if (has_c) {
          const float cv = pr.c_trans ? pr.C[(long long)b * pr.sc + (long long)gj * pr.ldc + pi]
                                      : pr.C[(long long)b * pr.sc + (long long)pi * pr.ldc + gj];
          o = fmaf(beta, cv, o);
        }
        if (pr.check_finite) bad |= !isfinite(o);
        if (pr.d_trans)
          pr.D[(long long)b * pr.sd + (long long)gj * pr.ldd + pi] = o;
        else
          pr.D[(long long)b * pr.sd + (long long)pi * pr.ldd + gj] = o;
        if (pr.D2)
          pr.D2[(long long)b * pr.s2 + (long long)pi * pr.ld2 + gj] = o + ((gi == gj && gi < pr.diag_limit) ? pr.gamma : 0.f);
        if (mirror) {
          pr.D[(long long)b * pr.sd + (long long)gj * pr.ldd + gi] = o;
          if (pr.D2) pr.D2[(long long)b * pr.s2 + (long long)gj * pr.ld2 + gi] = o;
        }
      }
    }
    if (bad) bad_any = 1;
    __syncthreads();
    if (tid == 0 && bad_any) set_status(P.status, GNS_DEVST_NONFINITE);
    __syncthreads();
  }
}

}  // namespace simt

int gemm_launch_f32(const GemmOp* ops, int nops, const uint32_t* dep_masks, int* counters, int32_t* dev_status,
                    void* stream, std::string* err) {
  (void)counters;
  for (int i = 0; i < nops; ++i)
    if (dep_masks && dep_masks[i]) {
      *err = "internal: the fp32 GEMM launches dependent products one by one";
      return GNS_ERR_INVALID;
    }
  using namespace simt;
  if (nops < 1 || nops > MAX_PROB) {
    *err = "internal: bad number of grouped products";
    return GNS_ERR_INVALID;
  }
  Params P;
  memset(&P, 0, sizeof(P));
  int tiles = 0;
  for (int i = 0; i < nops; ++i) {
    const GemmOp& o = ops[i];
    if (o.scale_part) {
      *err = "internal: the fp32 path takes the norm scale as a finished array";
      return GNS_ERR_UNSUPPORTED;
    }
    Problem& pr = P.prob[i];
    pr.A = static_cast<const float*>(o.A.ptr);
    pr.lda = o.A.ld;
    pr.sa = o.A.stride;
    pr.a_mn = o.a_mn;
    pr.B = static_cast<const float*>(o.B.ptr);
    pr.ldb = o.B.ld;
    pr.sb = o.B.stride;
    pr.b_mn = o.b_mn;
    pr.M = (int)o.M;
    pr.N = (int)o.N;
    pr.K = (int)o.K;
    pr.am = (int)(o.a_mn ? o.A.cols : o.A.rows);
    pr.ak = (int)std::min<int64_t>(o.K, o.a_mn ? o.A.rows : o.A.cols);
    pr.bn = (int)(o.b_mn ? o.B.cols : o.B.rows);
    pr.bk = (int)std::min<int64_t>(o.K, o.b_mn ? o.B.rows : o.B.cols);
    pr.tiles_m = (int)((o.M + T - 1) / T);
    pr.tiles_n = (int)((o.N + T - 1) / T);
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
    pr.C = static_cast<const float*>(o.C.ptr);
    pr.ldc = o.C.ld;
    pr.sc = o.C.stride;
    pr.c_trans = o.c_trans;
    pr.D = static_cast<float*>(o.D.ptr);
    pr.ldd = o.D.ld;
    pr.sd = o.D.stride;
    pr.d_trans = o.d_trans;
    pr.D2 = static_cast<float*>(o.D2.ptr);
    pr.ld2 = o.D2.ld;
    pr.s2 = o.D2.stride;
    pr.diag_limit = (int)o.diag_limit;
    pr.row_map = o.row_map;
    pr.rms = o.row_map_stride;
    pr.check_finite = o.check_finite;
  }
  P.nprob = nops;
  P.total_tiles = tiles;
  P.status = dev_status;
  if (tiles == 0) return GNS_OK;
  const int grid = std::min(tiles, device_sm_count() * 8);
  gemm_kernel<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(P);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    *err = std::string("fp32 GEMM launch: ") + cudaGetErrorString(e);
    return GNS_ERR_CUDA;
  }
  return GNS_OK;
}

}  // namespace gns
