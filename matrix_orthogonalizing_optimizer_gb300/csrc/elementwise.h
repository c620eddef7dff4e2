// Internal launchers of the HBM-bound kernels of libgns (elementwise.cu).
#pragma once

#include <stdint.h>

#include <string>

#include "gemm.h"

namespace gns {

constexpr int NPART = 32;           // parts per matrix of a deterministic reduction
constexpr int KEY_DIGITS = 10;      // base-2^32 digits of an exact l1 key (320 bits)
constexpr int MAX_SELECT_N = 65536; // largest selection dimension (shared-memory state)

int launch_sumsq(gns_dtype dt, const MatRef& X, int64_t count, float* partials, void* stream, std::string* err);
int launch_momentum(const MatRef& M, const MatRef& G, int64_t count, float mu, int mode, float* partials,
                    void* stream, std::string* err);
int launch_finalize_norm(const float* partials, int64_t count, float eps, float* inv, void* stream, std::string* err);
int launch_frac_add_keys(const MatRef& M, const MatRef& G, int64_t count, int trans, unsigned long long* keys,
                         int* nf, void* stream, std::string* err);
int launch_keys_only(const MatRef& M, int64_t count, int trans, unsigned long long* keys, int* nf, void* stream,
                     std::string* err);
int launch_select_topk(unsigned long long* keys, const int* nf, int64_t n, int64_t k, int64_t count, int* idx,
                       void* stream, std::string* err);
int launch_gather(const MatRef& M, int64_t count, int trans, const int* idx, int64_t k, const MatRef& X,
                  float* partials, void* stream, std::string* err);
int launch_decay_selected(const MatRef& M, int64_t count, int trans, const int* idx, int64_t k, float mu,
                          void* stream, std::string* err);
int launch_scale_unselected(const MatRef& W, int64_t count, int trans, const int* idx, int64_t k, float factor,
                            void* stream, std::string* err);
int launch_scatter_update(const MatRef& W, const MatRef& O, int64_t count, int trans, const int* idx, int64_t k,
                          float alpha, float beta, void* stream, std::string* err);
int launch_axpby(gns_dtype dt, const MatRef& W, const MatRef& Y, int64_t count, float alpha, float beta, void* stream,
                 std::string* err);
int launch_copy(gns_dtype dt, const MatRef& D, const MatRef& S, int64_t count, void* stream, std::string* err);

}  // namespace gns
