// C ABI of libgns (include/gns.h): argument validation, workspace planning and the stage
// sequences of standard and Gram Newton-Schulz, the Muon step and the Dion3 fractional
// update, expressed as batched GEMM launches (gemm_tc.cu / gemm_simt.cu) and HBM-bound
// kernels (elementwise.cu). No host synchronisation and no device allocation happen here.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstring>
#include <string>
#include <vector>

#include "../../include/gns.h"
#include "chain_small.h"
#include "elementwise.h"
#include "gemm.h"

namespace gns {

static thread_local std::string g_err;

static int fail(int code, const std::string& msg) {
  g_err = msg;
  return code;
}

static int64_t round_up(int64_t v, int64_t a) { return (v + a - 1) / a * a; }

int set_error(int code, const std::string& msg) { return fail(code, msg); }

// ---------------------------------------------------------------------------------------
// instrumentation (gns_profile_set / gns_profile_query)

struct ProfileState {
  void** events = nullptr;
  int capacity = 0;
  int gemm = 0;
  int all = 0;
};
static thread_local ProfileState g_prof;

// A failed event record (e.g. an invalid handle) is cleared so it cannot surface as the
// error of a later launch; instrumentation never fails a computation.
static void record_event(void* ev, void* stream) {
  if (cudaEventRecord(static_cast<cudaEvent_t>(ev), static_cast<cudaStream_t>(stream)) != cudaSuccess)
    (void)cudaGetLastError();
}

void profile_gemm_begin(void* stream) {
  if (g_prof.events && g_prof.gemm < g_prof.capacity) record_event(g_prof.events[2 * g_prof.gemm], stream);
}

void profile_gemm_end(void* stream) {
  if (g_prof.events && g_prof.gemm < g_prof.capacity) record_event(g_prof.events[2 * g_prof.gemm + 1], stream);
  ++g_prof.gemm;
  ++g_prof.all;
}

void profile_count_launch() { ++g_prof.all; }

// ---------------------------------------------------------------------------------------
// programs of dependent GEMMs

static bool op_conflict(const GemmOp& first, const GemmOp& later) {
  const void* w1[2] = {first.D.ptr, first.D2.ptr};
  const void* r1[3] = {first.A.ptr, first.B.ptr, first.C.ptr};
  const void* w2[2] = {later.D.ptr, later.D2.ptr};
  const void* r2[3] = {later.A.ptr, later.B.ptr, later.C.ptr};
  for (const void* w : w1) {
    if (!w) continue;
    for (const void* r : r2)
      if (r == w) return true;  // read after write
    for (const void* x : w2)
      if (x == w) return true;  // write after write
  }
  for (const void* r : r1) {
    if (!r) continue;
    for (const void* x : w2)
      if (x == r) return true;  // write after read
  }
  return false;
}

int gemm_program(gns_dtype dt, const GemmOp* ops, int nops, int* counters, int32_t* dev_status, void* stream,
                 std::string* err, bool counters_zeroed) {
  if (dt == GNS_F32) {
    for (int i = 0; i < nops; ++i) {
      int rc = gemm_launch(dt, ops + i, 1, dev_status, stream, err);
      if (rc) return rc;
    }
    return GNS_OK;
  }
  // upper-stored symmetric buffers: what a product with upper_out wrote
  std::vector<GemmOp> prog = with_types(dt, ops, nops);
  std::vector<const void*> upper;
  for (int j = 0; j < nops; ++j) {
    GemmOp& o = prog[j];
    for (const void* u : upper) {
      if (o.A.ptr == u) o.a_upper = 1;
      if (o.B.ptr == u) o.b_upper = 1;
    }
    if (o.upper_out && o.sym) {
      upper.push_back(o.D.ptr);
      if (o.D2.ptr) upper.push_back(o.D2.ptr);
    }
  }
  ops = prog.data();
  for (int base = 0; base < nops; base += kMaxProgramOps) {
    const int n = std::min(kMaxProgramOps, nops - base);
    uint32_t masks[kMaxProgramOps];
    uint32_t closure[kMaxProgramOps];  // every op an op waits for, directly or through others
    for (int j = 0; j < n; ++j) {
      masks[j] = 0;
      for (int i = 0; i < j; ++i)
        if (op_conflict(ops[base + i], ops[base + j])) masks[j] |= 1u << i;
      closure[j] = masks[j];
      for (int i = 0; i < j; ++i)
        if ((masks[j] >> i) & 1u) closure[j] |= closure[i];
      // transitive reduction: when op k (waited for) has itself waited for op i, op i's
      // completion for the same matrix is implied and need not be checked again
      uint32_t red = masks[j];
      for (int i = 0; i < j; ++i) {
        if (!((masks[j] >> i) & 1u)) continue;
        for (int k = i + 1; k < j; ++k)
          if (((masks[j] >> k) & 1u) && ((closure[k] >> i) & 1u)) {
            red &= ~(1u << i);
            break;
          }
      }
      masks[j] = red;
    }
    profile_gemm_begin(stream);
    int rc = gemm_launch_tc(ops + base, n, masks, counters, dev_status, stream, err, counters_zeroed && base == 0);
    profile_gemm_end(stream);
    if (rc) return rc;
  }
  return GNS_OK;
}

constexpr int64_t PAD = 128;  // padding of the n x n workspace matrices (tile size)

// ---------------------------------------------------------------------------------------
// workspace arena: the same planning code computes sizes (base == nullptr) and pointers

struct Arena {
  uint8_t* base = nullptr;
  size_t off = 0;
  void* take(size_t bytes) {
    off = (size_t)round_up((int64_t)off, 256);
    void* p = base ? base + off : nullptr;
    off += bytes;
    return p;
  }
};

// A workspace batch of `count` matrices with `rows_alloc` allocated rows, of which `rows`
// are valid: tensor maps and epilogues see `rows`, so the rows beyond read as zero.
static MatRef ws_mat(Arena& a, int64_t count, int64_t rows_alloc, int64_t rows, int64_t cols, int64_t ld,
                     size_t es) {
  MatRef m;
  m.rows = rows;
  m.cols = cols;
  m.ld = ld;
  m.stride = rows_alloc * ld;
  m.ptr = a.take((size_t)(count * m.stride) * es);
  return m;
}

static MatRef to_ref(const gns_batch& b) {
  MatRef m;
  m.ptr = b.ptr;
  m.ld = b.ld;
  m.stride = b.count > 1 ? b.stride : b.rows * b.ld;
  m.rows = b.rows;
  m.cols = b.cols;
  return m;
}

// ---------------------------------------------------------------------------------------
// validation

static size_t elem_size(gns_dtype dt) { return dt == GNS_F32 ? 4 : 2; }

static int check_batch(const gns_batch* b, gns_dtype dt, const char* name) {
  if (!b) return fail(GNS_ERR_INVALID, std::string(name) + ": null batch descriptor");
  const int64_t al = dt == GNS_F32 ? 4 : 8;
  if (!b->ptr) return fail(GNS_ERR_INVALID, std::string(name) + ": null data pointer");
  if (b->count < 1 || b->rows < 1 || b->cols < 1)
    return fail(GNS_ERR_INVALID, std::string(name) + ": count, rows and cols must be >= 1");
  // launch-grid limits: the matrix index and the smaller dimension run along grid y or z
  // (at most 65535 blocks), the larger dimension along y in tiles of at least 64
  if (b->count > 65535 || std::min(b->rows, b->cols) > 65535 || std::max(b->rows, b->cols) > 65535LL * 64)
    return fail(GNS_ERR_INVALID, std::string(name) +
                                     ": dimension too large (count and the smaller dimension at most 65535, the "
                                     "larger at most 4194240)");
  if (b->ld < b->cols) return fail(GNS_ERR_INVALID, std::string(name) + ": ld < cols");
  if (b->ld % al) return fail(GNS_ERR_UNSUPPORTED, std::string(name) + ": ld must be a multiple of 16 bytes");
  if (reinterpret_cast<uintptr_t>(b->ptr) % 16)
    return fail(GNS_ERR_UNSUPPORTED, std::string(name) + ": pointer must be 16-byte aligned");
  if (b->count > 1) {
    if (b->stride % al) return fail(GNS_ERR_UNSUPPORTED, std::string(name) + ": stride must be a multiple of 16 bytes");
    if (b->stride < b->rows * b->ld) return fail(GNS_ERR_INVALID, std::string(name) + ": stride < rows * ld");
  }
  return GNS_OK;
}

static int check_ns(const gns_ns_params* ns) {
  if (!ns) return fail(GNS_ERR_INVALID, "null ns params");
  if (ns->T < 1 || ns->T > GNS_MAX_T) return fail(GNS_ERR_INVALID, "T must be in [1, 16]");
  const uint32_t allowed = ns->T >= 2 ? (((1u << ns->T) - 1u) & ~1u) : 0u;
  if (ns->restart_mask & ~allowed)
    return fail(GNS_ERR_INVALID, "restart_mask bits must lie in [1, T-1] (restart after iteration i)");
  if (!(ns->eps >= 0.f) || !std::isfinite(ns->eps)) return fail(GNS_ERR_INVALID, "eps must be finite and >= 0");
  for (int t = 0; t < ns->T; ++t)
    if (!std::isfinite(ns->a[t]) || !std::isfinite(ns->b[t]) || !std::isfinite(ns->c[t]))
      return fail(GNS_ERR_INVALID, "coefficients must be finite");
  if (!(ns->safety > 0.f) || !std::isfinite(ns->safety))
    return fail(GNS_ERR_INVALID, "safety must be finite and > 0 (1 = no safety factor)");
  return GNS_OK;
}

// The schedule actually run: the safety factor of Dion3 appendix B.2.2, p_t(x / s), folded
// into the coefficients (a / s, b / s^3, c / s^5), computed in double and rounded once.
static gns_ns_params effective_ns(const gns_ns_params& ns) {
  gns_ns_params e = ns;
  const double s = ns.safety;
  if (s != 1.0)
    for (int t = 0; t < ns.T; ++t) {
      e.a[t] = (float)((double)ns.a[t] / s);
      e.b[t] = (float)((double)ns.b[t] / (s * s * s));
      e.c[t] = (float)((double)ns.c[t] / (s * s * s * s * s));
    }
  e.safety = 1.f;
  return e;
}

static bool same_shape(const gns_batch& a, const gns_batch& b) {
  return a.count == b.count && a.rows == b.rows && a.cols == b.cols;
}

// ---------------------------------------------------------------------------------------
// the oriented matrix X (n x m, n <= m) that one group orthogonalizes

struct Src {
  MatRef mat;        // physical storage
  int trans = 0;     // X = mat^T
  bool user = true;  // scaled by inv (user data) or already normalised (workspace)
};

// X as the A operand (or B operand of X X^T): X(i,k)
static void as_rows(const Src& s, MatRef* m, int* mn) {
  *m = s.mat;
  *mn = s.trans;
}
// X as the B operand of Q X: B(j,k) = X[k][j]
static void as_right(const Src& s, MatRef* m, int* mn) {
  *m = s.mat;
  *mn = s.trans ? 0 : 1;
}

// Final write: D = alpha' (Q X) + beta C with C = D (when has_c), optional row map.
// out_dt: element type of D (and C) when it differs from the products' (-1 = the same).
struct Final {
  MatRef D;
  int out_dt = -1;
  int d_trans = 0;
  float alpha = 1.f;
  float beta = 0.f;
  bool has_c = false;
  const int32_t* row_map = nullptr;
  int64_t rms = 0;
  int check_finite = 1;
};

// Groups of small matrices (oriented X at most 128 x 512) run whole in the on-chip chain
// kernel (chain_small.cu): one CTA per matrix, every product on one SM.
static bool chain_ok(bool gram, gns_dtype dt, const Src& src, int64_t n, int64_t m, const gns_ns_params* ns,
                     const Final& fin) {
  return fin.row_map == nullptr && chain_supported(gram, dt, n, m, src.trans, ns);
}

// One chain-kernel group: X as the source describes it, the result as the final write does.
// inv: per-matrix 1/(||X||_F + eps), or null to have the kernel sum the norm itself.
static ChainGroup chain_group(gns_dtype dt, const Src& src, int64_t B, int64_t n, int64_t m, const float* inv,
                              const Final& fin) {
  ChainGroup g;
  g.x = src.mat;
  g.xt = src.trans;
  g.B = B;
  g.n = n;
  g.m = m;
  g.inv = src.user ? inv : nullptr;
  g.D = fin.D;
  g.d_f16 = (fin.out_dt < 0 ? dt : (gns_dtype)fin.out_dt) == GNS_F16;
  g.d_trans = fin.d_trans;
  g.alpha = fin.alpha;
  g.beta = fin.beta;
  g.has_c = fin.has_c;
  return g;
}

// Chain-kernel groups collected over a call and launched together (one launch carries up to
// eight groups, so a small group's tail does not leave the chip idle until the next group's
// launch): one list per (algorithm, product type).
struct ChainBatch {
  ChainCall calls[2][2];  // [gram][fp16]
  void add(bool gram, gns_dtype dt, bool user, const gns_ns_params* ns, const ChainGroup& g) {
    ChainCall& c = calls[gram ? 1 : 0][dt == GNS_F16 ? 1 : 0];
    c.gram = gram;
    c.dt = dt;
    c.x_user = user;
    c.ns = ns;
    c.eps = ns->eps;
    c.groups.push_back(g);
  }
  int launch(int32_t* st, void* stream) {
    for (auto& row : calls)
      for (ChainCall& c : row) {
        if (c.groups.empty()) continue;
        c.status = st;
        c.stream = stream;
        std::string err;
        const int rc = launch_chain(c, &err);
        if (rc) return fail(rc, err);
      }
    return GNS_OK;
  }
};

static int run_chain(bool gram, gns_dtype dt, const Src& src, int64_t B, int64_t n, int64_t m,
                     const gns_ns_params* ns, const float* inv, const Final& fin, int32_t* st, void* stream) {
  ChainBatch cb;
  cb.add(gram, dt, src.user, ns, chain_group(dt, src, B, n, m, inv, fin));
  return cb.launch(st, stream);
}

struct GramBufs {
  float* partials = nullptr;
  float* inv = nullptr;
  int* counters = nullptr;
  MatRef R, Z, RZ, Q[2], X[2];
  int64_t np = 0;
};

struct StdBufs {
  float* partials = nullptr;
  float* inv = nullptr;
  int* counters = nullptr;
  MatRef A, Bm, X[2];
  int64_t np = 0;
};

static int popcount32(uint32_t v) {
  int c = 0;
  while (v) {
    c += v & 1u;
    v >>= 1;
  }
  return c;
}

static void plan_gram(Arena& a, int64_t B, int64_t n, int64_t m, gns_dtype dt, const gns_ns_params* ns, GramBufs* g,
                      bool with_norm) {
  const size_t es = elem_size(dt);
  g->np = round_up(n, PAD);
  const int64_t ldx = round_up(m, 8);
  if (with_norm) {
    g->partials = static_cast<float*>(a.take(sizeof(float) * NPART * B));
    g->inv = static_cast<float*>(a.take(sizeof(float) * B));
  }
  g->counters = static_cast<int*>(a.take(sizeof(int) * kMaxProgramOps * B));
  g->R = ws_mat(a, B, g->np, g->np, g->np, g->np, es);
  g->Z = ws_mat(a, B, g->np, g->np, g->np, g->np, es);
  g->RZ = ws_mat(a, B, g->np, g->np, g->np, g->np, es);
  g->Q[0] = ws_mat(a, B, g->np, g->np, g->np, g->np, es);
  g->Q[1] = ws_mat(a, B, g->np, g->np, g->np, g->np, es);
  const int nr = popcount32(ns->restart_mask);
  for (int i = 0; i < std::min(nr, 2); ++i) {
    g->X[i] = ws_mat(a, B, g->np, n, m, ldx, es);
  }
}

static void plan_std(Arena& a, int64_t B, int64_t n, int64_t m, gns_dtype dt, StdBufs* s, bool with_norm) {
  const size_t es = elem_size(dt);
  s->np = round_up(n, PAD);
  const int64_t ldx = round_up(m, 8);
  if (with_norm) {
    s->partials = static_cast<float*>(a.take(sizeof(float) * NPART * B));
    s->inv = static_cast<float*>(a.take(sizeof(float) * B));
  }
  s->counters = static_cast<int*>(a.take(sizeof(int) * kMaxProgramOps * B));
  s->A = ws_mat(a, B, s->np, s->np, s->np, s->np, es);
  s->Bm = ws_mat(a, B, s->np, s->np, s->np, s->np, es);
  s->X[0] = ws_mat(a, B, s->np, n, m, ldx, es);
  s->X[1] = ws_mat(a, B, s->np, n, m, ldx, es);
}

static GemmOp sym_op(const MatRef& A, int a_mn, const MatRef& Bm, int b_mn, int64_t K, int64_t np, int64_t B,
                     float alpha, int alpha_pow, const float* scale, const MatRef* C, float beta, const MatRef& D) {
  GemmOp o;
  o.A = A;
  o.a_mn = a_mn;
  o.B = Bm;
  o.b_mn = b_mn;
  o.M = o.N = np;
  o.K = K;
  o.batch = B;
  o.sym = 1;
  o.alpha = alpha;
  o.alpha_pow = alpha_pow;
  o.scale = scale;
  if (C) {
    o.C = *C;
    o.beta = beta;
  }
  o.D = D;
  return o;
}

// The Frobenius-norm scale 1 / (||X_b||_F + eps) of a group's products: the finished array
// (inv), or the per-matrix partial sums of squares the tensor-core GEMM forms it from (part),
// in which case the kernel that wrote them also zeroed the GEMM's completion counters.
struct NormScale {
  const float* inv = nullptr;
  const float* part = nullptr;
  float eps = 0.f;
  bool counters_zeroed = false;  // the group's GEMM completion counters are already zero
};

// Smallest oriented row count n whose groups take the scale from the partial sums: the GEMM
// forms it per scaled tile (a 128-byte line of partial sums per matrix); on smaller matrices,
// whose products are one short tile per matrix, that costs more than the finalize launch it
// saves (measured: the 1-CTA tile paths of n = 32 .. 256 slower by a few per cent).
constexpr int64_t kPartScaleMinN = 512;

static void set_scale(GemmOp* o, const NormScale& sc) {
  o->scale = sc.inv;
  if (sc.part) {
    o->scale_part = sc.part;
    o->scale_npart = NPART;
    o->scale_eps = sc.eps;
  }
}

// Dion3 Algorithm 3 on one group (B matrices, oriented X = n x m). sc: the norm scale of X
// (user data), already computed on the stream or to be formed by the GEMM.
static int run_gram(gns_dtype dt, const Src& src, int64_t B, int64_t n, int64_t m, const gns_ns_params* ns,
                    const GramBufs& g, const NormScale& sc, const Final& fin, int32_t* st, void* stream) {
  const float* inv = sc.inv;
  if (chain_ok(true, dt, src, n, m, ns, fin)) {
    if (!inv) return fail(GNS_ERR_UNSUPPORTED, "internal: the chain kernel takes the norm scale as an array");
    return run_chain(true, dt, src, B, n, m, ns, inv, fin, st, stream);
  }
  std::string err;
  const int64_t np = g.np;
  std::vector<GemmOp> prog;  // the whole sequence, in program order
  auto launch = [&](const GemmOp* ops, int nops) -> int {
    for (int i = 0; i < nops; ++i) prog.push_back(ops[i]);
    return GNS_OK;
  };
  int rc;
  Src X = src;
  // R_0 = X X^T (scaled by inv^2), the first Gram product of Algorithm 3
  {
    MatRef xa;
    int mn;
    as_rows(X, &xa, &mn);
    GemmOp o = sym_op(xa, mn, xa, mn, m, np, B, 1.f, X.user ? 2 : 0, nullptr, nullptr, 0.f, g.R);
    if (X.user) set_scale(&o, sc);
    if ((rc = launch(&o, 1))) return rc;
  }
  bool q_id = true;
  int qc = 0;
  int nx = 0;
  const int T = ns->T;
  for (int t = 1; t <= T; ++t) {
    const float a = ns->a[t - 1], b = ns->b[t - 1], c = ns->c[t - 1];
    if (t > 1 && ((ns->restart_mask >> (t - 1)) & 1u)) {
      // restart: X <- Q X; R <- X X^T; Q <- I
      MatRef xb;
      int bmn;
      as_right(X, &xb, &bmn);
      GemmOp o;
      o.A = g.Q[qc];
      o.a_mn = 0;
      o.B = xb;
      o.b_mn = bmn;
      o.M = n;
      o.N = m;
      o.K = np;
      o.batch = B;
      o.alpha = 1.f;
      o.alpha_pow = X.user ? 1 : 0;
      if (X.user) set_scale(&o, sc);
      MatRef xd = g.X[nx & 1];
      o.D = xd;
      if ((rc = launch(&o, 1))) return rc;
      ++nx;
      X.mat = xd;
      X.trans = 0;
      X.user = false;
      GemmOp r = sym_op(xd, 0, xd, 0, m, np, B, 1.f, 0, nullptr, nullptr, 0.f, g.R);
      if ((rc = launch(&r, 1))) return rc;
      q_id = true;
    }
    // Z = b R + c R^2 (a_t I is never added to Z, appendix B.2.3)
    GemmOp oz = sym_op(g.R, 0, g.R, 1, np, np, B, c, 0, nullptr, &g.R, b, g.Z);
    if (q_id) {
      // the Q update with Q_{t-1} = I: Q_t = Z_t + a_t I, written by the same launch
      oz.D2 = g.Q[qc];
      oz.gamma = a;
      oz.diag_limit = n;
    }
    if ((rc = launch(&oz, 1))) return rc;
    const bool r_needed = t < T && !((ns->restart_mask >> t) & 1u);
    GemmOp ops[2];
    int nops = 0;
    if (!q_id) {
      // Q_t = Q_{t-1} Z_t + a_t Q_{t-1}
      ops[nops++] = sym_op(g.Q[qc], 0, g.Z, 1, np, np, B, 1.f, 0, nullptr, &g.Q[qc], a, g.Q[1 - qc]);
    }
    if (r_needed) {
      // RZ_t = R_{t-1} Z_t + a_t R_{t-1}
      ops[nops++] = sym_op(g.R, 0, g.Z, 1, np, np, B, 1.f, 0, nullptr, &g.R, a, g.RZ);
    }
    if (nops && (rc = launch(ops, nops))) return rc;
    if (!q_id) qc = 1 - qc;
    if (r_needed) {
      // R_t = Z_t RZ_t + a_t RZ_t
      GemmOp orr = sym_op(g.Z, 0, g.RZ, 1, np, np, B, 1.f, 0, nullptr, &g.RZ, a, g.R);
      if ((rc = launch(&orr, 1))) return rc;
    }
    q_id = false;
  }
  // X <- Q_T X, written (or added) to the final destination
  {
    MatRef xb;
    int bmn;
    as_right(X, &xb, &bmn);
    GemmOp o;
    o.A = g.Q[qc];
    o.a_mn = 0;
    o.B = xb;
    o.b_mn = bmn;
    o.M = n;
    o.N = m;
    o.K = np;
    o.batch = B;
    o.alpha = fin.alpha;
    o.alpha_pow = X.user ? 1 : 0;
    if (X.user) set_scale(&o, sc);
    o.D = fin.D;
    o.d_trans = fin.d_trans;
    o.c_dt = o.d_dt = fin.out_dt;
    if (fin.has_c) {
      o.C = fin.D;
      o.c_trans = fin.d_trans;
      o.beta = fin.beta;
    }
    o.row_map = fin.row_map;
    o.row_map_stride = fin.rms;
    o.check_finite = fin.check_finite;
    if ((rc = launch(&o, 1))) return rc;
  }
  for (GemmOp& o : prog) o.upper_out = o.sym;  // internal symmetric buffers: upper tiles only
  rc = gemm_program(dt, prog.data(), (int)prog.size(), g.counters, st, stream, &err, sc.counters_zeroed);
  return rc ? fail(rc, err) : GNS_OK;
}

// Dion3 Algorithm 1 with symmetric products (sec. 2.3). Writes X_T to fin.D (direct mode,
// fin.has_c must be false) or, when to_ws, leaves it in the returned workspace buffer.
static int run_std(gns_dtype dt, const Src& src, int64_t B, int64_t n, int64_t m, const gns_ns_params* ns,
                   const StdBufs& s, const float* inv, const Final* fin, MatRef* result, int32_t* st, void* stream) {
  std::string err;
  const int64_t np = s.np;
  std::vector<GemmOp> prog;  // the whole sequence, in program order
  auto launch = [&](const GemmOp* ops, int nops) -> int {
    for (int i = 0; i < nops; ++i) prog.push_back(ops[i]);
    return GNS_OK;
  };
  int rc;
  Src X = src;
  for (int t = 1; t <= ns->T; ++t) {
    const float a = ns->a[t - 1], b = ns->b[t - 1], c = ns->c[t - 1];
    const int sp = X.user ? 1 : 0;
    MatRef xa;
    int amn;
    as_rows(X, &xa, &amn);
    // A = X X^T
    GemmOp oa = sym_op(xa, amn, xa, amn, m, np, B, 1.f, 2 * sp, inv, nullptr, 0.f, s.A);
    if ((rc = launch(&oa, 1))) return rc;
    // B = b A + c A^2
    GemmOp ob = sym_op(s.A, 0, s.A, 1, np, np, B, c, 0, nullptr, &s.A, b, s.Bm);
    if ((rc = launch(&ob, 1))) return rc;
    // X <- a X + B X
    MatRef xb;
    int bmn;
    as_right(X, &xb, &bmn);
    GemmOp ox;
    ox.A = s.Bm;
    ox.a_mn = 0;
    ox.B = xb;
    ox.b_mn = bmn;
    ox.K = np;
    ox.batch = B;
    ox.alpha = 1.f;
    ox.alpha_pow = sp;
    ox.scale = inv;
    ox.C = X.mat;
    ox.c_trans = X.trans;
    ox.beta = a;
    ox.beta_pow = sp;
    const bool last = t == ns->T;
    if (last && fin) {
      ox.M = n;
      ox.N = m;
      ox.D = fin->D;
      ox.d_trans = fin->d_trans;
      ox.d_dt = fin->out_dt;
      ox.check_finite = fin->check_finite;
    } else {
      ox.M = n;
      ox.N = m;
      ox.D = s.X[(t - 1) & 1];
      ox.check_finite = last;
    }
    if ((rc = launch(&ox, 1))) return rc;
    X.mat = ox.D;
    X.trans = 0;
    X.user = false;
    if (last && result) *result = ox.D;
  }
  for (GemmOp& o : prog) o.upper_out = o.sym;  // internal symmetric buffers: upper tiles only
  rc = gemm_program(dt, prog.data(), (int)prog.size(), s.counters, st, stream, &err);
  return rc ? fail(rc, err) : GNS_OK;
}

// ---------------------------------------------------------------------------------------
// per-op planning shared by sizing and execution

struct GroupShape {
  int64_t B, rows, cols, n, m;
  int trans;
};

static GroupShape shape_of(const gns_batch& x) {
  GroupShape g;
  g.B = x.count;
  g.rows = x.rows;
  g.cols = x.cols;
  g.trans = x.rows > x.cols;
  g.n = std::min(x.rows, x.cols);
  g.m = std::max(x.rows, x.cols);
  return g;
}

static int64_t frac_k(float frac, int64_t n) {
  int64_t k = (int64_t)std::ceil((double)frac * (double)n - 1e-9);
  return std::max<int64_t>(1, std::min<int64_t>(k, n));
}

// The flavour one step runs: Periodic Row-wise Muon (Scaling Muon for DiTs eq. (7)) takes
// Newton-Schulz on the refresh steps t mod K == 0 and RowNorm on the others.
static int step_flavor(const gns_muon_params& mp) {
  if (mp.flavor == GNS_FLAVOR_PERIODIC) {
    const int64_t t = mp.step, K = mp.period;
    return ((t % K) + K) % K == 0 ? GNS_FLAVOR_MUON : GNS_FLAVOR_ROWNORM;
  }
  return mp.flavor;
}

// Workspace of one group of a Muon step; the same code sizes (Arena without base) and
// places the buffers.
struct MuonBufs {
  bool frac = false, use_std = false;
  int flavor = GNS_FLAVOR_MUON;
  gns_dtype nsdt = GNS_BF16;
  int64_t k = 0;
  StdBufs sb;
  GramBufs gb;
  MatRef x16;                          // normalised fp16 copy of M (or of M[S])
  unsigned long long* keys = nullptr;  // frac: selection
  int* nf = nullptr;
  int* idx = nullptr;
  MatRef xs, os;                       // frac: M[S] and O before the scatter
  MatRef o;                            // dense NorMuon: O (oriented, bf16)
  float* s = nullptr;                  // NorMuon / RowNorm: row sums of squares
  float* r = nullptr;                  // and row scales
  float* part = nullptr;               // RowNorm of a tall matrix: column partial sums
  float* colpart = nullptr;            // frac, tall: per-block sums of squares of the column gather
  int64_t ncolpart = 0;
};

static void plan_muon(Arena& a, const GroupShape& sh, const gns_muon_params& mp, const gns_ns_params* ns,
                      MuonBufs* mb) {
  mb->flavor = step_flavor(mp);
  mb->nsdt = mp.ns_dtype == GNS_F16 ? GNS_F16 : GNS_BF16;
  mb->frac = mp.frac < 1.f;
  const int64_t B = sh.B, n = sh.n, m = sh.m;
  const int64_t ldm = round_up(m, 8);
  if (mb->flavor == GNS_FLAVOR_ROWNORM) {
    mb->s = static_cast<float*>(a.take(sizeof(float) * B * n));
    mb->r = static_cast<float*>(a.take(sizeof(float) * B * n));
    if (sh.trans) mb->part = static_cast<float*>(a.take(sizeof(float) * B * NPART * n));
    return;
  }
  const bool normuon = mb->flavor == GNS_FLAVOR_NORMUON;
  if (!mb->frac) {
    mb->use_std = n == m;
    if (mb->use_std)
      plan_std(a, B, n, m, mb->nsdt, &mb->sb, true);
    else
      plan_gram(a, B, n, m, mb->nsdt, ns, &mb->gb, true);
    if (mb->nsdt == GNS_F16)
      mb->x16 = ws_mat(a, B, sh.rows, sh.rows, sh.cols, round_up(sh.cols, 8), 2);
    if (normuon) {
      mb->o = ws_mat(a, B, n, n, m, ldm, 2);
      mb->s = static_cast<float*>(a.take(sizeof(float) * B * n));
      mb->r = static_cast<float*>(a.take(sizeof(float) * B * n));
    }
    return;
  }
  const int64_t k = frac_k(mp.frac, n);
  mb->k = k;
  mb->keys = static_cast<unsigned long long*>(a.take(sizeof(unsigned long long) * KEY_DIGITS * n * B));
  mb->nf = static_cast<int*>(a.take(sizeof(int) * n * B));
  mb->idx = static_cast<int*>(a.take(sizeof(int) * k * B));
  if (sh.trans) {
    mb->ncolpart = gather_cols_blocks(k, sh.rows);
    mb->colpart = static_cast<float*>(a.take(sizeof(float) * B * mb->ncolpart));
  }
  mb->xs = ws_mat(a, B, round_up(k, PAD), k, m, ldm, 2);
  // O gets its own buffer only where the update cannot ride on the last product's epilogue:
  // NorMuon (its row statistics need O first) and the columns of a tall matrix, where the
  // Muon flavour stores O transposed (m x k) for the column scatter
  if (normuon)
    mb->os = ws_mat(a, B, k, k, m, ldm, 2);
  else if (sh.trans)
    mb->os = ws_mat(a, B, m, m, k, round_up(k, 8), 2);
  if (mb->nsdt == GNS_F16) mb->x16 = ws_mat(a, B, round_up(k, PAD), k, m, ldm, 2);
  plan_gram(a, B, k, m, mb->nsdt, ns, &mb->gb, true);
  if (normuon) {
    mb->s = static_cast<float*>(a.take(sizeof(float) * B * k));
    mb->r = static_cast<float*>(a.take(sizeof(float) * B * k));
  }
}

}  // namespace gns

using namespace gns;

extern "C" {

int gns_version(void) { return GNS_VERSION; }

int gns_profile_set(void** events, int capacity) {
  if (events && capacity < 0) return fail(GNS_ERR_INVALID, "negative capacity");
  g_prof.events = events;
  g_prof.capacity = events ? capacity : 0;
  g_prof.gemm = 0;
  g_prof.all = 0;
  return GNS_OK;
}

int gns_profile_query(int* gemm_launches, int* all_launches) {
  if (gemm_launches) *gemm_launches = g_prof.gemm;
  if (all_launches) *all_launches = g_prof.all;
  return GNS_OK;
}

const char* gns_status_string(int s) {
  switch (s) {
    case GNS_OK: return "GNS_OK";
    case GNS_ERR_INVALID: return "GNS_ERR_INVALID";
    case GNS_ERR_UNSUPPORTED: return "GNS_ERR_UNSUPPORTED";
    case GNS_ERR_WORKSPACE: return "GNS_ERR_WORKSPACE";
    case GNS_ERR_CUDA: return "GNS_ERR_CUDA";
    default: return "GNS_UNKNOWN_STATUS";
  }
}

int gns_last_error(char* buf, size_t len) {
  if (buf && len) {
    const size_t n = std::min(len - 1, g_err.size());
    memcpy(buf, g_err.data(), n);
    buf[n] = 0;
  }
  return (int)g_err.size();
}

void gns_ns_params_default(gns_ns_params* p) {
  if (!p) return;
  memset(p, 0, sizeof(*p));
  p->T = 5;
  for (int t = 0; t < 5; ++t) {
    p->a[t] = 3.4445f;
    p->b[t] = -4.7750f;
    p->c[t] = 2.0315f;
  }
  p->restart_mask = 1u << 2;
  p->eps = 1e-7f;
  p->safety = 1.f;
}

static int check_muon(const gns_muon_params& mp) {
  if (!(mp.frac > 0.f) || mp.frac > 1.f) return fail(GNS_ERR_INVALID, "frac must be in (0, 1]");
  if (!std::isfinite(mp.lr) || !std::isfinite(mp.momentum) || !std::isfinite(mp.weight_decay) ||
      !std::isfinite(mp.scale))
    return fail(GNS_ERR_INVALID, "muon params must be finite");
  if (mp.flavor < GNS_FLAVOR_MUON || mp.flavor > GNS_FLAVOR_PERIODIC) return fail(GNS_ERR_INVALID, "unknown flavor");
  if (mp.ns_dtype != GNS_BF16 && mp.ns_dtype != GNS_F16)
    return fail(GNS_ERR_INVALID, "ns_dtype must be GNS_BF16 or GNS_F16");
  if (mp.flavor == GNS_FLAVOR_NORMUON) {
    if (!(mp.beta2 >= 0.f && mp.beta2 < 1.f)) return fail(GNS_ERR_INVALID, "NorMuon beta2 must be in [0, 1)");
    if (!(mp.norm_eps > 0.f) || !std::isfinite(mp.norm_eps))
      return fail(GNS_ERR_INVALID, "NorMuon norm_eps must be finite and > 0");
  }
  if (mp.flavor == GNS_FLAVOR_ROWNORM || mp.flavor == GNS_FLAVOR_PERIODIC) {
    if (mp.frac < 1.f) return fail(GNS_ERR_UNSUPPORTED, "RowNorm flavours are dense steps (frac = 1)");
    if (!(mp.norm_eps > 0.f) || !std::isfinite(mp.norm_eps))
      return fail(GNS_ERR_INVALID, "RowNorm norm_eps must be finite and > 0");
    if (!(mp.rownorm_gamma > 0.f) || !std::isfinite(mp.rownorm_gamma))
      return fail(GNS_ERR_INVALID, "rownorm_gamma must be finite and > 0");
  }
  if (mp.flavor == GNS_FLAVOR_PERIODIC && mp.period < 1) return fail(GNS_ERR_INVALID, "period must be >= 1");
  return GNS_OK;
}

static int plan_op(gns_op op, const gns_batch* x, int ngroups, gns_dtype dt, const gns_ns_params* ns,
                   const gns_muon_params* mp, Arena& a) {
  if (!x || ngroups < 1) return fail(GNS_ERR_INVALID, "need at least one batch");
  if (dt != GNS_BF16 && dt != GNS_F32 && dt != GNS_F16) return fail(GNS_ERR_INVALID, "unknown dtype");
  if (op != GNS_OP_FRAC_SELECT) {
    int rc = check_ns(ns);
    if (rc) return rc;
  }
  for (int gi = 0; gi < ngroups; ++gi) {
    int rc = check_batch(&x[gi], dt, "x");
    if (rc) return rc;
    GroupShape s = shape_of(x[gi]);
    if (op == GNS_OP_GRAM_NS) {
      if (s.n == s.m) {
        StdBufs sb;
        plan_std(a, s.B, s.n, s.m, dt, &sb, true);
      } else {
        GramBufs gb;
        plan_gram(a, s.B, s.n, s.m, dt, ns, &gb, true);
      }
    } else if (op == GNS_OP_NS_STANDARD) {
      StdBufs sb;
      plan_std(a, s.B, s.n, s.m, dt, &sb, true);
    } else if (op == GNS_OP_MUON_STEP) {
      if (!mp) return fail(GNS_ERR_INVALID, "null muon params");
      if (dt != GNS_BF16) return fail(GNS_ERR_UNSUPPORTED, "Muon steps take bf16 W, G, M");
      if ((rc = check_muon(*mp))) return rc;
      MuonBufs mb;
      plan_muon(a, s, *mp, ns, &mb);
    } else if (op == GNS_OP_FRAC_SELECT) {
      a.take(sizeof(unsigned long long) * KEY_DIGITS * s.n * s.B);
      a.take(sizeof(int) * s.n * s.B);
      a.take(sizeof(float) * NPART * s.B);
    } else {
      return fail(GNS_ERR_INVALID, "unknown op");
    }
  }
  return GNS_OK;
}

}  // extern "C"

namespace gns {
// Workspace bytes of a request in *need, returning the planner's status (and setting the last
// error) when the request is invalid or unsupported.
int plan_workspace(gns_op op, const gns_batch* x, int ngroups, gns_dtype dtype, const gns_ns_params* ns,
                   const gns_muon_params* muon, size_t* need) {
  Arena a;
  *need = 0;
  const int rc = plan_op(op, x, ngroups, dtype, ns, muon, a);
  if (rc) return rc;
  *need = a.off + 256;
  return GNS_OK;
}
}  // namespace gns

extern "C" {

size_t gns_workspace_size(gns_op op, const gns_batch* x, int ngroups, gns_dtype dtype, const gns_ns_params* ns,
                          const gns_muon_params* muon) {
  size_t need = 0;
  return plan_workspace(op, x, ngroups, dtype, ns, muon, &need) ? 0 : need;
}

static int check_ws(void* ws, size_t ws_bytes, size_t need) {
  if (need && !ws) return fail(GNS_ERR_WORKSPACE, "null workspace");
  if (reinterpret_cast<uintptr_t>(ws) % 256) return fail(GNS_ERR_WORKSPACE, "workspace must be 256-byte aligned");
  if (ws_bytes < need)
    return fail(GNS_ERR_WORKSPACE, "workspace too small: need " + std::to_string(need) + " bytes");
  return GNS_OK;
}

static int ns_common(bool gram, const gns_batch* x, const gns_batch* out, int ngroups, gns_dtype dt,
                     const gns_ns_params* ns, void* ws, size_t ws_bytes, int32_t* st, void* stream) {
  if (!out) return fail(GNS_ERR_INVALID, "null out");
  const gns_op op = gram ? GNS_OP_GRAM_NS : GNS_OP_NS_STANDARD;
  size_t need = 0;
  int rc = plan_workspace(op, x, ngroups, dt, ns, nullptr, &need);
  if (rc) return rc;
  rc = check_ws(ws, ws_bytes, need);
  if (rc) return rc;
  for (int gi = 0; gi < ngroups; ++gi) {
    if ((rc = check_batch(&out[gi], dt, "out"))) return rc;
    if (!same_shape(x[gi], out[gi])) return fail(GNS_ERR_INVALID, "out must have the shape of x");
    if (x[gi].ptr == out[gi].ptr) return fail(GNS_ERR_INVALID, "out may not alias x");
  }
  Arena a;
  a.base = static_cast<uint8_t*>(ws);
  std::string err;
  const gns_ns_params nse = effective_ns(*ns);
  ns = &nse;
  ChainBatch chains;
  for (int gi = 0; gi < ngroups; ++gi) {
    GroupShape s = shape_of(x[gi]);
    Src src;
    src.mat = to_ref(x[gi]);
    src.trans = s.trans;
    Final fin;
    fin.D = to_ref(out[gi]);
    fin.d_trans = s.trans;
    const bool g_alg = gram && s.n != s.m;
    if (chain_ok(g_alg, dt, src, s.n, s.m, ns, fin)) {
      // launched with the call's other small groups below; the norm is summed inside the
      // kernel, from the X it holds on chip
      chains.add(g_alg, dt, true, ns, chain_group(dt, src, s.B, s.n, s.m, nullptr, fin));
      continue;
    }
    if (g_alg) {
      GramBufs gb;
      plan_gram(a, s.B, s.n, s.m, dt, ns, &gb, true);
      NormScale sc;
      if (dt != GNS_F32 && s.n >= kPartScaleMinN) {
        // the GEMM forms the scale from the partial sums; their kernel zeroes its counters
        sc.part = gb.partials;
        sc.eps = ns->eps;
        sc.counters_zeroed = true;
        if ((rc = launch_sumsq(dt, src.mat, s.B, gb.partials, stream, &err, gb.counters, kMaxProgramOps * (int)s.B)))
          return fail(rc, err);
      } else {
        sc.inv = gb.inv;
        if ((rc = launch_sumsq(dt, src.mat, s.B, gb.partials, stream, &err))) return fail(rc, err);
        if ((rc = launch_finalize_norm(gb.partials, s.B, ns->eps, gb.inv, stream, &err))) return fail(rc, err);
      }
      if ((rc = run_gram(dt, src, s.B, s.n, s.m, ns, gb, sc, fin, st, stream))) return rc;
    } else {
      StdBufs sb;
      plan_std(a, s.B, s.n, s.m, dt, &sb, true);
      if ((rc = launch_sumsq(dt, src.mat, s.B, sb.partials, stream, &err))) return fail(rc, err);
      if ((rc = launch_finalize_norm(sb.partials, s.B, ns->eps, sb.inv, stream, &err))) return fail(rc, err);
      if ((rc = run_std(dt, src, s.B, s.n, s.m, ns, sb, sb.inv, &fin, nullptr, st, stream))) return rc;
    }
  }
  return chains.launch(st, stream);
}

int gns_gram_ns_batched(const gns_batch* x, const gns_batch* out, int ngroups, gns_dtype dtype,
                        const gns_ns_params* ns, void* ws, size_t ws_bytes, int32_t* dev_status, void* stream) {
  return ns_common(true, x, out, ngroups, dtype, ns, ws, ws_bytes, dev_status, stream);
}

int gns_ns_standard_batched(const gns_batch* x, const gns_batch* out, int ngroups, gns_dtype dtype,
                            const gns_ns_params* ns, void* ws, size_t ws_bytes, int32_t* dev_status, void* stream) {
  return ns_common(false, x, out, ngroups, dtype, ns, ws, ws_bytes, dev_status, stream);
}

int gns_sym_gemm_xxt(const gns_batch* x, const gns_batch* c, float alpha, float beta, gns_dtype dt,
                     int32_t* dev_status, void* stream) {
  int rc;
  if ((rc = check_batch(x, dt, "x")) || (rc = check_batch(c, dt, "c"))) return rc;
  if (c->count != x->count || c->rows != x->rows || c->cols != x->rows)
    return fail(GNS_ERR_INVALID, "c must be count x rows x rows of x");
  if (x->ptr == c->ptr) return fail(GNS_ERR_INVALID, "c may not alias x");
  MatRef xm = to_ref(*x), cm = to_ref(*c);
  GemmOp o = sym_op(xm, 0, xm, 0, x->cols, x->rows, x->count, alpha, 0, nullptr, beta != 0.f ? &cm : nullptr, beta, cm);
  std::string err;
  rc = gemm_launch(dt, &o, 1, dev_status, stream, &err);
  return rc ? fail(rc, err) : GNS_OK;
}

int gns_sym_gemm(const gns_batch* a, const gns_batch* b, const gns_batch* c, const gns_batch* d, float alpha,
                 float beta, gns_dtype dt, int32_t* dev_status, void* stream) {
  int rc;
  if ((rc = check_batch(a, dt, "a")) || (rc = check_batch(b, dt, "b")) || (rc = check_batch(d, dt, "d"))) return rc;
  const int64_t n = a->rows;
  if (a->cols != n || b->rows != n || b->cols != n || d->rows != n || d->cols != n || b->count != a->count ||
      d->count != a->count)
    return fail(GNS_ERR_INVALID, "a, b, d must be count x n x n");
  if (beta != 0.f) {
    if (!c) return fail(GNS_ERR_INVALID, "c is required when beta != 0");
    if ((rc = check_batch(c, dt, "c"))) return rc;
    if (!same_shape(*c, *d)) return fail(GNS_ERR_INVALID, "c must have the shape of d");
  }
  if (d->ptr == a->ptr || d->ptr == b->ptr) return fail(GNS_ERR_INVALID, "d may not alias a or b");
  MatRef am = to_ref(*a), bm = to_ref(*b), dm = to_ref(*d);
  MatRef cm;
  if (beta != 0.f) cm = to_ref(*c);
  GemmOp o = sym_op(am, 0, bm, 1, n, n, a->count, alpha, 0, nullptr, beta != 0.f ? &cm : nullptr, beta, dm);
  std::string err;
  rc = gemm_launch(dt, &o, 1, dev_status, stream, &err);
  return rc ? fail(rc, err) : GNS_OK;
}

int gns_sym_poly_update(const gns_batch* R, const gns_batch* Q, const gns_batch* Z, const gns_batch* RZ,
                        const gns_batch* q_scratch, float a, float b, float c, int q_is_identity, int skip_r,
                        gns_dtype dt, int32_t* dev_status, void* stream) {
  int rc;
  if ((rc = check_batch(R, dt, "R")) || (rc = check_batch(Q, dt, "Q")) || (rc = check_batch(Z, dt, "Z")) ||
      (rc = check_batch(RZ, dt, "RZ")))
    return rc;
  const int64_t n = R->rows;
  if (R->cols != n || !same_shape(*R, *Q) || !same_shape(*R, *Z) || !same_shape(*R, *RZ))
    return fail(GNS_ERR_INVALID, "R, Q, Z, RZ must be count x n x n");
  if (!q_is_identity) {
    if ((rc = check_batch(q_scratch, dt, "q_scratch"))) return rc;
    if (!same_shape(*R, *q_scratch)) return fail(GNS_ERR_INVALID, "q_scratch must be count x n x n");
  }
  const int64_t B = R->count;
  MatRef r = to_ref(*R), q = to_ref(*Q), z = to_ref(*Z), rz = to_ref(*RZ);
  std::string err;
  GemmOp oz = sym_op(r, 0, r, 1, n, n, B, c, 0, nullptr, &r, b, z);
  if (q_is_identity) {
    oz.D2 = q;
    oz.gamma = a;
    oz.diag_limit = n;
  }
  if ((rc = gemm_launch(dt, &oz, 1, dev_status, stream, &err))) return fail(rc, err);
  GemmOp ops[2];
  int nops = 0;
  MatRef qs;
  if (!q_is_identity) {
    qs = to_ref(*q_scratch);
    ops[nops++] = sym_op(q, 0, z, 1, n, n, B, 1.f, 0, nullptr, &q, a, qs);
  }
  if (!skip_r) ops[nops++] = sym_op(r, 0, z, 1, n, n, B, 1.f, 0, nullptr, &r, a, rz);
  if (nops && (rc = gemm_launch(dt, ops, nops, dev_status, stream, &err))) return fail(rc, err);
  if (!q_is_identity && (rc = launch_copy(dt, q, qs, B, stream, &err))) return fail(rc, err);
  if (!skip_r) {
    GemmOp orr = sym_op(z, 0, rz, 1, n, n, B, 1.f, 0, nullptr, &rz, a, r);
    if ((rc = gemm_launch(dt, &orr, 1, dev_status, stream, &err))) return fail(rc, err);
  }
  return GNS_OK;
}

int gns_muon_step(const gns_batch* W, const gns_batch* G, const gns_batch* M, const gns_batch* V, int ngroups,
                  const gns_muon_params* mp, const gns_ns_params* ns, void* ws, size_t ws_bytes,
                  int32_t* dev_status, void* stream) {
  if (!W || !G || !M || !mp) return fail(GNS_ERR_INVALID, "null argument");
  if (ngroups < 1) return fail(GNS_ERR_INVALID, "need at least one batch");
  int rc;
  if ((rc = check_muon(*mp))) return rc;
  const bool normuon = step_flavor(*mp) == GNS_FLAVOR_NORMUON;
  if (normuon && !V) return fail(GNS_ERR_INVALID, "NorMuon needs the second-moment batches V");
  for (int gi = 0; gi < ngroups; ++gi) {
    if ((rc = check_batch(&W[gi], GNS_BF16, "W")) || (rc = check_batch(&G[gi], GNS_BF16, "G")) ||
        (rc = check_batch(&M[gi], GNS_BF16, "M")))
      return rc;
    if (!same_shape(W[gi], G[gi]) || !same_shape(W[gi], M[gi]))
      return fail(GNS_ERR_INVALID, "W, G, M must have equal shapes");
    if (W[gi].ptr == G[gi].ptr || W[gi].ptr == M[gi].ptr || G[gi].ptr == M[gi].ptr)
      return fail(GNS_ERR_INVALID, "W, G, M may not alias");
    if (normuon) {
      if ((rc = check_batch(&V[gi], GNS_F32, "V"))) return rc;
      if (V[gi].count != M[gi].count || V[gi].rows != 1 || V[gi].cols != std::min(M[gi].rows, M[gi].cols))
        return fail(GNS_ERR_INVALID, "V must be count x 1 x min(rows, cols) (fp32)");
      if (V[gi].ptr == W[gi].ptr || V[gi].ptr == G[gi].ptr || V[gi].ptr == M[gi].ptr)
        return fail(GNS_ERR_INVALID, "V may not alias W, G or M");
    }
  }
  size_t need = 0;
  if ((rc = plan_workspace(GNS_OP_MUON_STEP, M, ngroups, GNS_BF16, ns, mp, &need))) return rc;
  if ((rc = check_ws(ws, ws_bytes, need))) return rc;
  const gns_ns_params nse = effective_ns(*ns);
  ns = &nse;
  Arena a;
  a.base = static_cast<uint8_t*>(ws);
  std::string err;
  const float lr = mp->lr, mu = mp->momentum;
  const float decay = 1.f - mp->lr * mp->weight_decay;
  const float step_scale = -lr * mp->scale;
  ChainBatch chains;
  for (int gi = 0; gi < ngroups; ++gi) {
    GroupShape s = shape_of(M[gi]);
    MatRef mm = to_ref(M[gi]), gm = to_ref(G[gi]), wm = to_ref(W[gi]);
    MatRef vm;
    if (normuon) vm = to_ref(V[gi]);
    MuonBufs mb;
    plan_muon(a, s, *mp, ns, &mb);
    if (mb.flavor == GNS_FLAVOR_ROWNORM) {
      // Scaling Muon for DiTs eq. (5), (7) off a refresh step: M <- mu M + G;
      // W <- (1 - lr wd) W - lr scale gamma R_eps(M) on the oriented rows of M
      if (!s.trans && rownorm_fused_supported(s.cols)) {
        if ((rc = launch_rownorm_fused_rows(mm, gm, wm, s.B, mu, mp->rownorm_gamma, mp->norm_eps, step_scale, decay,
                                            stream, &err)))
          return fail(rc, err);
        continue;
      }
      if ((rc = launch_momentum(mm, gm, s.B, mu, 0, nullptr, stream, &err))) return fail(rc, err);
      if (!s.trans)
        rc = launch_row_sumsq(mm, s.rows, s.cols, s.B, mb.s, stream, &err);
      else
        rc = launch_col_sumsq(mm, s.B, mb.part, mb.s, stream, &err);
      if (rc) return fail(rc, err);
      if ((rc = launch_rownorm_scale(mb.s, s.B * s.n, mp->rownorm_gamma, mp->norm_eps, mb.r, stream, &err)))
        return fail(rc, err);
      if ((rc = launch_rowscale_update(wm, mm, mb.r, s.B, s.trans, step_scale, decay, stream, &err)))
        return fail(rc, err);
      continue;
    }
    if (!mb.frac) {
      // Muon, eq. (1) (NorMuon, eq. (2)): M <- mu M + G; O = polar(M); W <- (1 - lr wd) W - lr scale O
      float* partials = mb.use_std ? mb.sb.partials : mb.gb.partials;
      float* inv = mb.use_std ? mb.sb.inv : mb.gb.inv;
      Src src;
      src.mat = mm;
      src.trans = s.trans;
      Final fin;
      fin.out_dt = GNS_BF16;
      if (normuon) {
        fin.D = mb.o;  // O, oriented
      } else if (!mb.use_std) {
        fin.D = wm;  // the weight update in the last product's epilogue
        fin.d_trans = s.trans;
        fin.alpha = step_scale;
        fin.beta = decay;
        fin.has_c = true;
      }
      Final fs = fin;  // the standard-NS flavour's final write
      if (mb.use_std && !normuon) {
        fs.D = wm;
        fs.d_trans = s.trans;
        fs.alpha = step_scale;
        fs.beta = decay;
        fs.has_c = true;
      }
      // bf16 Gram NS on the tile path (n >= kPartScaleMinN): the GEMM forms the norm scale from
      // the momentum pass's partial sums (no finalize launch), and that pass zeroes the GEMM's
      // completion counters
      const bool part_scale = !mb.use_std && mb.nsdt == GNS_BF16 && s.n >= kPartScaleMinN &&
                              !chain_ok(true, mb.nsdt, src, s.n, s.m, ns, fin);
      if ((rc = launch_momentum(mm, gm, s.B, mu, 0, partials, stream, &err, part_scale ? mb.gb.counters : nullptr,
                                part_scale ? kMaxProgramOps * (int)s.B : 0)))
        return fail(rc, err);
      if (!part_scale && (rc = launch_finalize_norm(partials, s.B, ns->eps, inv, stream, &err))) return fail(rc, err);
      if (mb.nsdt == GNS_F16) {
        // Dion3 Algorithm 3, normalise then cast: the normalised momentum, rounded once to float16
        if ((rc = launch_cast_scaled(mb.x16, mm, inv, s.B, stream, &err))) return fail(rc, err);
        src.mat = mb.x16;
        src.user = false;
      }
      if (!normuon) {
        const bool g_alg = !mb.use_std;
        const Final& ff = g_alg ? fin : fs;
        if (chain_ok(g_alg, mb.nsdt, src, s.n, s.m, ns, ff)) {
          // the orthogonalization and update of this small group run in the chain kernel,
          // launched once for all such groups of the call after the loop
          chains.add(g_alg, mb.nsdt, src.user, ns, chain_group(mb.nsdt, src, s.B, s.n, s.m, inv, ff));
          continue;
        }
      }
      if (mb.use_std && chain_ok(false, mb.nsdt, src, s.n, s.m, ns, fs)) {
        if ((rc = run_chain(false, mb.nsdt, src, s.B, s.n, s.m, ns, inv, fs, dev_status, stream))) return rc;
      } else if (mb.use_std) {
        MatRef xt;
        if ((rc = run_std(mb.nsdt, src, s.B, s.n, s.m, ns, mb.sb, inv, normuon ? &fin : nullptr, &xt, dev_status,
                          stream)))
          return rc;
        if (!normuon) {
          MatRef xv = xt;
          xv.rows = s.n;
          if ((rc = launch_axpby(GNS_BF16, wm, xv, s.B, step_scale, decay, stream, &err, mb.nsdt)))
            return fail(rc, err);
        }
      } else {
        NormScale sc;
        if (part_scale) {
          sc.part = partials;
          sc.eps = ns->eps;
          sc.counters_zeroed = true;
        } else {
          sc.inv = inv;
        }
        if ((rc = run_gram(mb.nsdt, src, s.B, s.n, s.m, ns, mb.gb, sc, fin, dev_status, stream))) return rc;
      }
      if (normuon) {
        // eq. (2): second moments of the rows of O, row scaling, Frobenius rescale, update
        if ((rc = launch_row_sumsq(mb.o, s.n, s.m, s.B, mb.s, stream, &err))) return fail(rc, err);
        if ((rc = launch_normuon_rows(mb.s, vm, nullptr, s.n, s.m, s.B, mp->beta2, mp->norm_eps, mb.r, stream,
                                      &err)))
          return fail(rc, err);
        if ((rc = launch_scatter_update(wm, mb.o, s.B, s.trans, nullptr, s.n, step_scale, decay, stream, &err,
                                        mb.r)))
          return fail(rc, err);
      }
      continue;
    }
    // Dion3 Algorithm 4
    const int64_t k = mb.k;
    // M <- M + G, with the exact l1 keys of the oriented rows
    if ((rc = launch_frac_add_keys(mm, gm, s.B, s.trans, mb.keys, mb.nf, stream, &err))) return fail(rc, err);
    // selection
    if ((rc = launch_select_topk(mb.keys, mb.nf, s.n, k, s.B, mb.idx, stream, &err))) return fail(rc, err);
    // gather M[S, :] and its Frobenius norm; the error feedback (M[S] <- mu M[S]) rides
    // on the same pass: M[S] is not read again
    if ((rc = launch_gather(mm, s.B, s.trans, mb.idx, k, mb.xs, mb.gb.partials, stream, &err, true, mu, mb.colpart)))
      return fail(rc, err);
    if ((rc = s.trans ? launch_finalize_norm(mb.colpart, s.B, ns->eps, mb.gb.inv, stream, &err, mb.ncolpart)
                      : launch_finalize_norm(mb.gb.partials, s.B, ns->eps, mb.gb.inv, stream, &err)))
      return fail(rc, err);
    // weight decay on the rows that are not updated below
    if (decay != 1.f && (rc = launch_scale_unselected(wm, s.B, s.trans, mb.idx, k, decay, mb.nf, stream, &err)))
      return fail(rc, err);
    // O = polar(M[S])
    Src src;
    src.mat = mb.xs;
    src.trans = 0;
    if (mb.nsdt == GNS_F16) {
      if ((rc = launch_cast_scaled(mb.x16, mb.xs, mb.gb.inv, s.B, stream, &err))) return fail(rc, err);
      src.mat = mb.x16;
      src.user = false;
    }
    Final fin;
    fin.out_dt = GNS_BF16;
    const bool fused = !normuon && !s.trans;
    if (fused) {
      // W[S] <- (1 - lr wd) W[S] - lr scale O in the last product's epilogue (Dion3 sec. 6,
      // "Weight update"): rows of O go to the selected rows of W, fp32 arithmetic, one rounding
      fin.D = wm;
      fin.alpha = step_scale;
      fin.beta = decay;
      fin.has_c = true;
      fin.row_map = mb.idx;
      fin.rms = k;
    } else {
      fin.D = mb.os;
      fin.d_trans = normuon ? 0 : 1;  // the tall Muon flavour's column scatter reads O transposed
    }
    NormScale sc;
    sc.inv = mb.gb.inv;
    if ((rc = run_gram(mb.nsdt, src, s.B, k, s.m, ns, mb.gb, sc, fin, dev_status, stream))) return rc;
    if (fused) continue;
    if (!normuon) {
      // W[:, S] <- (1 - lr wd) W[:, S] - lr scale O^T, one rounding
      if ((rc = launch_scatter_update_cols_t(wm, mb.os, s.B, mb.idx, k, step_scale, decay, stream, &err)))
        return fail(rc, err);
      continue;
    }
    // NorMuon flavour: second moments of the selected rows, scaling, rescale
    if (normuon) {
      if ((rc = launch_row_sumsq(mb.os, k, s.m, s.B, mb.s, stream, &err))) return fail(rc, err);
      if ((rc = launch_normuon_rows(mb.s, vm, mb.idx, k, s.m, s.B, mp->beta2, mp->norm_eps, mb.r, stream, &err)))
        return fail(rc, err);
    }
    // W[S] <- (1 - lr wd) W[S] - lr scale O, one rounding
    if ((rc = launch_scatter_update(wm, mb.os, s.B, s.trans, mb.idx, k, step_scale, decay, stream, &err,
                                    normuon ? mb.r : nullptr)))
      return fail(rc, err);
  }
  return chains.launch(dev_status, stream);
}

int gns_selftest_bounded_wait(const int32_t* counter, int32_t target, uint32_t limit_us, int32_t* dev_status,
                              uint64_t* out, void* stream) {
  if (!counter || reinterpret_cast<uintptr_t>(counter) % 4) return fail(GNS_ERR_INVALID, "counter: null or unaligned");
  if (out && reinterpret_cast<uintptr_t>(out) % 8) return fail(GNS_ERR_INVALID, "out: unaligned");
  if (limit_us < 1 || limit_us > 2000000u) return fail(GNS_ERR_INVALID, "limit_us must be in [1, 2000000]");
  std::string err;
  int rc = launch_selftest_wait(counter, target, (uint64_t)limit_us * 1000ull, dev_status,
                                reinterpret_cast<unsigned long long*>(out), stream, &err);
  return rc ? fail(rc, err) : GNS_OK;
}

int gns_frac_row_select(const gns_batch* m, int k, int32_t* idx, const gns_batch* gathered, void* ws,
                        size_t ws_bytes, void* stream) {
  int rc;
  if ((rc = check_batch(m, GNS_BF16, "m"))) return rc;
  if (!idx) return fail(GNS_ERR_INVALID, "null idx");
  GroupShape s = shape_of(*m);
  if (k < 1 || k > s.n) return fail(GNS_ERR_INVALID, "k must be in [1, min(rows, cols)]");
  size_t need = gns_workspace_size(GNS_OP_FRAC_SELECT, m, 1, GNS_BF16, nullptr, nullptr);
  if ((rc = check_ws(ws, ws_bytes, need))) return rc;
  if (gathered) {
    if ((rc = check_batch(gathered, GNS_BF16, "gathered"))) return rc;
    if (gathered->count != s.B || gathered->rows != k || gathered->cols != s.m)
      return fail(GNS_ERR_INVALID, "gathered must be count x k x max(rows, cols)");
  }
  Arena a;
  a.base = static_cast<uint8_t*>(ws);
  auto* keys = static_cast<unsigned long long*>(a.take(sizeof(unsigned long long) * KEY_DIGITS * s.n * s.B));
  auto* nf = static_cast<int*>(a.take(sizeof(int) * s.n * s.B));
  auto* partials = static_cast<float*>(a.take(sizeof(float) * NPART * s.B));
  std::string err;
  MatRef mm = to_ref(*m);
  if ((rc = launch_keys_only(mm, s.B, s.trans, keys, nf, stream, &err))) return fail(rc, err);
  if ((rc = launch_select_topk(keys, nf, s.n, k, s.B, idx, stream, &err))) return fail(rc, err);
  if (gathered && (rc = launch_gather(mm, s.B, s.trans, idx, k, to_ref(*gathered), partials, stream, &err)))
    return fail(rc, err);
  return GNS_OK;
}

}  // extern "C"
