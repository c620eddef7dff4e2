// Internal interface of the batched GEMM launchers of libgns (not part of the C ABI).
//
// Every product in the library has the form
//     D = alpha' * (A (x) B) + beta' * C          (per matrix b of a batch)
// with (A (x) B)[i][j] = sum_k A(i,k) B(j,k), i < M, j < N, k < K, where
//     A(i,k) = a_mn ? A[k][i] : A[i][k]      (physical row-major matrices)
//     B(j,k) = b_mn ? B[k][j] : B[j][k]
// so an ordinary product A * Bmat is b_mn = 1 with B = Bmat, and X X^T is A = B = X with
// a_mn = b_mn = 0. alpha' = alpha * scale[b]^alpha_pow, beta' = beta * scale[b]^beta_pow.
// With scale_part set instead (tensor-core kernel only), scale[b] = 1 / (sqrt(s) + scale_eps),
// s the sum of the scale_npart = 32 partial sums scale_part[b * 32 + p] (16-byte aligned) by a
// fixed pairwise tree in fp32 (fp64 where that overflows): the Frobenius-norm scale, formed by
// the GEMM from the norm pass's partial sums.
// C and D are read / written at (i, j) (or at (j, i) when c_trans / d_trans), with the
// row index i replaced by row_map[b * row_map_stride + i] when row_map is set.
// sym: M == N and only tiles with tile_row <= tile_col are computed; each off-diagonal tile
// is also written to its mirrored position (j, i); diagonal tiles are written once.
// D2 (optional, same layout as D): D + gamma * I on the diagonal entries i == j < diag_limit.
// Element types: A and B share ab_dt; C and D (with D2) have c_dt and d_dt; -1 means the
// dtype of the call that launches the op (gemm_launch / gemm_program). The tensor-core
// kernel takes bf16 and fp16 in any combination of (ab, c, d); the fp32 path all fp32.
#pragma once

#include <vector>

#include <stdint.h>

#include <string>

#include "../../include/gns.h"

namespace gns {

struct MatRef {
  void* ptr = nullptr;  // element (0,0) of matrix 0
  int64_t ld = 0;       // elements between rows
  int64_t stride = 0;   // elements between matrices
  int64_t rows = 0;     // physical rows
  int64_t cols = 0;     // physical cols
};

struct GemmOp {
  MatRef A;
  int a_mn = 0;
  MatRef B;
  int b_mn = 0;
  int64_t M = 0, N = 0, K = 0, batch = 0;
  int sym = 0;
  float alpha = 1.f, beta = 0.f, gamma = 0.f;
  int alpha_pow = 0, beta_pow = 0;
  const float* scale = nullptr;
  const float* scale_part = nullptr;
  int scale_npart = 0;
  float scale_eps = 0.f;
  MatRef C;
  int c_trans = 0;
  MatRef D;
  int d_trans = 0;
  MatRef D2;
  int64_t diag_limit = 0;
  const int32_t* row_map = nullptr;
  int64_t row_map_stride = 0;
  int check_finite = 0;
  // bf16 kernel only: upper_out = this symmetric product stores its upper-triangle tiles
  // only (no mirrored copies); a_upper / b_upper = that operand is such an upper-stored
  // symmetric matrix, read transposed wherever a K slice falls below its diagonal.
  int upper_out = 0;
  int a_upper = 0, b_upper = 0;
  int ab_dt = -1, c_dt = -1, d_dt = -1;
};

// Copies of ops with every unset (-1) element type replaced by dt.
inline std::vector<GemmOp> with_types(gns_dtype dt, const GemmOp* ops, int nops) {
  std::vector<GemmOp> v(ops, ops + nops);
  for (GemmOp& o : v) {
    if (o.ab_dt < 0) o.ab_dt = dt;
    if (o.c_dt < 0) o.c_dt = dt;
    if (o.d_dt < 0) o.d_dt = dt;
  }
  return v;
}

// Enqueues ops as ONE launch. dep_masks[i] (nullable) names earlier ops of the same launch
// whose tiles of the same matrix must be complete before a tile of op i starts (the
// tensor-core kernel waits on per-(op, matrix) completion counters: `counters`, at least
// sum(batch) ints of device memory, reset by the launch unless counters_zeroed: then the
// kernel enqueued just before it on the stream has zeroed them). Without masks the ops must be
// mutually independent. A launch with an op that forms its scale from partial sums
// (scale_part) is a programmatic dependent launch: it may begin while the kernel before it on
// the stream ends, and reads and writes global memory only after that kernel has completed.
// Returns GNS_OK or an error status with *err set.
int gemm_launch_tc(const GemmOp* ops, int nops, const uint32_t* dep_masks, int* counters, int32_t* dev_status,
                   void* stream, std::string* err, bool counters_zeroed = false);
int gemm_launch_f32(const GemmOp* ops, int nops, const uint32_t* dep_masks, int* counters, int32_t* dev_status,
                    void* stream, std::string* err);

// Instrumentation (gns_profile_set): event records around GEMM launches, launch counts.
void profile_gemm_begin(void* stream);
void profile_gemm_end(void* stream);
void profile_count_launch();

// Independent ops as one launch.
inline int gemm_launch(gns_dtype dt, const GemmOp* ops, int nops, int32_t* dev_status, void* stream,
                       std::string* err) {
  const std::vector<GemmOp> typed = with_types(dt, ops, nops);
  profile_gemm_begin(stream);
  const int rc = dt != GNS_F32 ? gemm_launch_tc(typed.data(), nops, nullptr, nullptr, dev_status, stream, err)
                               : gemm_launch_f32(typed.data(), nops, nullptr, nullptr, dev_status, stream, err);
  profile_gemm_end(stream);
  return rc;
}

// Largest number of ops of one tensor-core launch.
constexpr int kMaxProgramOps = 24;

// A sequence of ops in program order (op j may read what op i < j wrote, or overwrite what
// it read). bf16 / fp16: as few launches as possible, dependencies between ops found from
// the buffers they read (A, B, C) and write (D, D2) and enforced per matrix inside the
// launch; fp32: one launch per op, ordered by the stream. `counters`: kMaxProgramOps * batch ints,
// already zero when counters_zeroed (see gemm_launch_tc).
int gemm_program(gns_dtype dt, const GemmOp* ops, int nops, int* counters, int32_t* dev_status, void* stream,
                 std::string* err, bool counters_zeroed = false);

// Number of SMs of the current device (cached per device).
int device_sm_count();

}  // namespace gns
