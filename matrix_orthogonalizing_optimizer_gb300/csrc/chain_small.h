// Internal interface of the on-chip chain kernel (chain_small.cu): Gram or standard
// Newton-Schulz for matrices whose oriented X has at most 128 rows and 512 columns, one CTA
// per matrix, every product of the chain on one SM. One launch carries up to eight shape
// groups (more are split over several launches).
#pragma once

#include <stdint.h>

#include <string>
#include <vector>

#include "gemm.h"

namespace gns {

// One shape group: count B of oriented n x m matrices X and their results.
struct ChainGroup {
  MatRef x;                    // the user's X (storage)
  int xt = 0;                  // X = storage^T (a tall matrix; Gram only)
  int64_t B = 0, n = 0, m = 0;
  const float* inv = nullptr;  // per-matrix 1/(||X||_F + eps), or null (summed in the kernel)
  // D = alpha * O + beta * D (has_c), O = the orthogonalized X, written at (i, j) or at (j, i)
  // when d_trans
  MatRef D;
  int d_f16 = 0;
  int d_trans = 0;
  float alpha = 1.f, beta = 0.f;
  bool has_c = false;
};

struct ChainCall {
  bool gram = true;           // Dion3 Algorithm 3 (else Algorithm 1)
  gns_dtype dt = GNS_BF16;    // element type of the products (bf16 or fp16)
  bool x_user = true;         // X not yet normalised: products are scaled by 1/(||X||_F + eps)
  const gns_ns_params* ns = nullptr;  // effective schedule (safety factor already folded in)
  float eps = 0.f;
  int check_finite = 1;
  std::vector<ChainGroup> groups;  // every group passes chain_supported; all or none carry inv
  int32_t* status = nullptr;
  void* stream = nullptr;
};

// Whether the chain kernel takes this group (shape, type, schedule length; the environment
// variable GNS_CHAIN_SMALL=0 turns it off).
bool chain_supported(bool gram, gns_dtype dt, int64_t n, int64_t m, int xt, const gns_ns_params* ns);

// Enqueues the groups (one launch per eight). Returns GNS_OK or an error status with *err set.
int launch_chain(const ChainCall& c, std::string* err);

}  // namespace gns
