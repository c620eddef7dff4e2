// Internal launchers of the HBM-bound kernels of libgns (elementwise.cu).
#pragma once

#include <stdint.h>

#include <string>

#include "gemm.h"

namespace gns {

constexpr int NPART = 32;           // parts per matrix of a deterministic reduction
constexpr int KEY_DIGITS = 10;      // base-2^32 digits of an exact l1 key (320 bits)
constexpr int MAX_SELECT_N = 65536; // largest selection dimension (shared-memory state)

// zero / nzero (optional): ints the kernel sets to 0 (the completion counters of the GEMM launch
// enqueued right after it, which then skips its own reset).
int launch_sumsq(gns_dtype dt, const MatRef& X, int64_t count, float* partials, void* stream, std::string* err,
                 int* zero = nullptr, int nzero = 0);
int launch_momentum(const MatRef& M, const MatRef& G, int64_t count, float mu, int mode, float* partials,
                    void* stream, std::string* err, int* zero = nullptr, int nzero = 0);
// npart: partials per matrix (NPART, or a gather's per-block sums, gather_cols_blocks).
int launch_finalize_norm(const float* partials, int64_t count, float eps, float* inv, void* stream, std::string* err,
                         int64_t npart = NPART);
// Blocks per matrix of the column gather of a tall matrix (k selected columns, rows rows):
// the per-block sums of squares it stores with bpart.
int64_t gather_cols_blocks(int64_t k, int64_t rows);
int launch_frac_add_keys(const MatRef& M, const MatRef& G, int64_t count, int trans, unsigned long long* keys,
                         int* nf, void* stream, std::string* err);
int launch_keys_only(const MatRef& M, int64_t count, int trans, unsigned long long* keys, int* nf, void* stream,
                     std::string* err);
int launch_select_topk(unsigned long long* keys, const int* nf, int64_t n, int64_t k, int64_t count, int* idx,
                       void* stream, std::string* err);
// decay: also M[S] <- bf16(mu * M[S]) in the same pass (Algorithm 4's error feedback).
// Columns of a tall M (trans): with bpart (gather_cols_blocks(k, rows) floats per matrix) the
// gather stores its per-block sums of squares there instead of filling partials by a second
// pass over X.
int launch_gather(const MatRef& M, int64_t count, int trans, const int* idx, int64_t k, const MatRef& X,
                  float* partials, void* stream, std::string* err, bool decay = false, float mu = 1.f,
                  float* bpart = nullptr);
// flags: count * n ints of scratch (n = rows, or cols when trans).
int launch_scale_unselected(const MatRef& W, int64_t count, int trans, const int* idx, int64_t k, float factor,
                            int* flags, void* stream, std::string* err);
// rs (nullable): per-row scale of O (NorMuon); idx NULL: every row, in order.
int launch_scatter_update(const MatRef& W, const MatRef& O, int64_t count, int trans, const int* idx, int64_t k,
                          float alpha, float beta, void* stream, std::string* err, const float* rs = nullptr);
// Columns idx of a tall W from the transpose of O (OT: len x k, len = rows of W):
// W[j][idx[i]] <- bf16(beta W + alpha OT[j][i]).
int launch_scatter_update_cols_t(const MatRef& W, const MatRef& OT, int64_t count, const int* idx, int64_t k,
                                 float alpha, float beta, void* stream, std::string* err);
// y_dt: type of Y when it differs from W's (bf16 W with fp16 Y); -1 = dt.
int launch_axpby(gns_dtype dt, const MatRef& W, const MatRef& Y, int64_t count, float alpha, float beta, void* stream,
                 std::string* err, gns_dtype y_dt = (gns_dtype)-1);
// s[b*k + i] = sum of squares of row i (of `cols` entries) of the bf16 batch X.
int launch_row_sumsq(const MatRef& X, int64_t k, int64_t cols, int64_t count, float* s, void* stream,
                     std::string* err);
// s[b*cols + c] = sum of squares of column c of the bf16 batch M; part: NPART * cols * count
// floats of scratch.
int launch_col_sumsq(const MatRef& M, int64_t count, float* part, float* s, void* stream, std::string* err);
// NorMuon second moments (V fp32, updated at rows idx or 0..k-1) and row scales r.
int launch_normuon_rows(const float* s, const MatRef& V, const int* idx, int64_t k, int64_t len, int64_t count,
                        float beta2, float eps, float* r, void* stream, std::string* err);
// Single-pass RowNorm step on the rows of a wide matrix (cols a multiple of 8, at most
// 16384): momentum, row norm and the scaled weight update in one kernel.
bool rownorm_fused_supported(int64_t cols);
int launch_rownorm_fused_rows(const MatRef& M, const MatRef& G, const MatRef& W, int64_t count, float mu, float gamma,
                              float eps, float alpha, float beta, void* stream, std::string* err);
// RowNorm scales r = gamma / max(sqrt(s), eps) over n entries.
int launch_rownorm_scale(const float* s, int64_t n, float gamma, float eps, float* r, void* stream,
                         std::string* err);
// W <- beta W + alpha r_q Y with q the row (trans 0) or column (trans 1) of each element.
int launch_rowscale_update(const MatRef& W, const MatRef& Y, const float* r, int64_t count, int trans, float alpha,
                           float beta, void* stream, std::string* err);
// X16 = fp16(inv[b] * M) in M's layout.
int launch_cast_scaled(const MatRef& X16, const MatRef& M, const float* inv, int64_t count, void* stream,
                       std::string* err);
int launch_copy(gns_dtype dt, const MatRef& D, const MatRef& S, int64_t count, void* stream, std::string* err);
// One block whose bounded waits (a completion counter, then an mbarrier phase nothing
// completes) run out after limit_ns each (gns_selftest_bounded_wait).
int launch_selftest_wait(const int* counter, int target, uint64_t limit_ns, int* status, unsigned long long* out,
                         void* stream, std::string* err);

}  // namespace gns
