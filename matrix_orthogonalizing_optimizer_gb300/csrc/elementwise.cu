// HBM-bound kernels of libgns: momentum update with fused Frobenius statistics, norm
// finalisation, exact l1 selection keys, top-k row selection, row gather / scatter /
// decay, and small batched copies.
//
// Reductions are deterministic: every matrix is split into a fixed number of parts
// (NPART), each part reduced by one block in a fixed order, and the parts summed in a
// fixed order. Selection keys are exact integers, so their reduction order cannot matter.
#include <algorithm>

#include "common.cuh"
#include "elementwise.h"

namespace gns {

// ---------------------------------------------------------------------------------------
// block reduction helpers

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Sum over a block of 256 threads in a fixed order (warp shuffles, then warp 0).
__device__ float block_sum_256(float v) {
  __shared__ float ws[8];
  v = warp_sum(v);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) ws[w] = v;
  __syncthreads();
  float t = 0.f;
  if (w == 0) {
    t = l < 8 ? ws[l] : 0.f;
    t = warp_sum(t);
  }
  return t;  // valid in thread 0
}

template <typename T>
__device__ __forceinline__ float to_f(T v);
template <>
__device__ __forceinline__ float to_f<float>(float v) {
  return v;
}
template <>
__device__ __forceinline__ float to_f<bf16>(bf16 v) {
  return __bfloat162float(v);
}
template <>
__device__ __forceinline__ float to_f<__half>(__half v) {
  return __half2float(v);
}

template <typename T>
__device__ __forceinline__ T from_f(float v);
template <>
__device__ __forceinline__ float from_f<float>(float v) {
  return v;
}
template <>
__device__ __forceinline__ bf16 from_f<bf16>(float v) {
  return __float2bfloat16_rn(v);
}
template <>
__device__ __forceinline__ __half from_f<__half>(float v) {
  return __float2half_rn(v);
}

// ---------------------------------------------------------------------------------------
// sum of squares per matrix (read only), partials[b * npart + part]

// The norm pass (sumsq_kernel, momentum_kernel) may also zero `nzero` ints at `zero` (the
// completion counters of the GEMM launch that follows it on the stream), and lets that launch
// begin while it finishes.
__device__ __forceinline__ void zero_and_release(int* zero, int nzero) {
  grid_dep_launch();
  if (zero && blockIdx.x == 0 && blockIdx.y == 0)
    for (int i = threadIdx.x; i < nzero; i += blockDim.x) zero[i] = 0;
}

// Rows start on 16-byte boundaries (ld and the base are 16-byte aligned), so each thread
// reads 16-byte vectors of VEC elements; a scalar tail covers cols % VEC.
template <typename T>
__global__ void sumsq_kernel(const T* X, long long ld, long long stride, int rows, int cols, int npart,
                             float* partials, int* zero, int nzero) {
  constexpr int VEC = 16 / sizeof(T);
  zero_and_release(zero, nzero);
  const int b = blockIdx.y, part = blockIdx.x;
  const int rp = (rows + npart - 1) / npart;
  const int r0 = part * rp, r1 = min(rows, r0 + rp);
  const T* Xb = X + (long long)b * stride;
  const int cvec = cols - cols % VEC;
  float acc = 0.f;
  for (int r = r0; r < r1; ++r) {
    const T* row = Xb + (long long)r * ld;
#pragma unroll 4
    for (int c = threadIdx.x * VEC; c < cvec; c += blockDim.x * VEC) {
      const uint4 u = *reinterpret_cast<const uint4*>(row + c);
      const T* e = reinterpret_cast<const T*>(&u);
#pragma unroll
      for (int q = 0; q < VEC; ++q) {
        const float v = to_f(e[q]);
        acc = fmaf(v, v, acc);
      }
    }
    for (int c = cvec + threadIdx.x; c < cols; c += blockDim.x) {
      const float v = to_f(row[c]);
      acc = fmaf(v, v, acc);
    }
  }
  const float s = block_sum_256(acc);
  if (threadIdx.x == 0) partials[(long long)b * npart + part] = s;
}

// Rows of a batch processed by one block each chunk of ROWS_PER_BLOCK rows, threads over
// 16-byte vectors of the row.
constexpr int ROWS_PER_BLOCK = 4;

// ---------------------------------------------------------------------------------------
// momentum: M <- mu * M + G (mode 0; fp32 product, fp32 sum, one bf16 rounding) or
// M <- M + G (mode 1), with the sum of squares of the stored new M in partials (when set).

__device__ __forceinline__ float mom(float m, float g, float mu, int mode) {
  return mode == 0 ? __fadd_rn(__fmul_rn(mu, m), g) : __fadd_rn(m, g);
}

__global__ void momentum_kernel(bf16* M, long long ldm, long long sm, const bf16* G, long long ldg, long long sg,
                                int rows, int cols, float mu, int mode, int npart, float* partials, int* zero,
                                int nzero) {
  zero_and_release(zero, nzero);
  const int b = blockIdx.y, part = blockIdx.x;
  const int rp = (rows + npart - 1) / npart;
  const int r0 = part * rp, r1 = min(rows, r0 + rp);
  bf16* Mb = M + (long long)b * sm;
  const bf16* Gb = G + (long long)b * sg;
  float acc = 0.f;
  const int cvec = cols & ~7;
  for (int r = r0; r < r1; ++r) {
    bf16* mr = Mb + (long long)r * ldm;
    const bf16* gr = Gb + (long long)r * ldg;
    for (int c = threadIdx.x * 8; c < cvec; c += blockDim.x * 8) {
      uint4 mv = *reinterpret_cast<const uint4*>(mr + c);
      const uint4 gv = *reinterpret_cast<const uint4*>(gr + c);
      bf16* me = reinterpret_cast<bf16*>(&mv);
      const bf16* ge = reinterpret_cast<const bf16*>(&gv);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const bf16 nv = f_to_bf16(mom(bf16_to_f(me[e]), bf16_to_f(ge[e]), mu, mode));
        me[e] = nv;
        const float f = bf16_to_f(nv);
        acc = fmaf(f, f, acc);
      }
      *reinterpret_cast<uint4*>(mr + c) = mv;
    }
    for (int c = cvec + threadIdx.x; c < cols; c += blockDim.x) {
      const bf16 nv = f_to_bf16(mom(bf16_to_f(mr[c]), bf16_to_f(gr[c]), mu, mode));
      mr[c] = nv;
      const float f = bf16_to_f(nv);
      acc = fmaf(f, f, acc);
    }
  }
  if (partials) {
    const float s = block_sum_256(acc);
    if (threadIdx.x == 0) partials[(long long)b * npart + part] = s;
  }
}

// inv[b] = 1 / (sqrt(sum of the npart partials) + eps) for many partials, one block of 256
// threads per matrix: thread t sums a contiguous run of partials in order (fp64), the runs
// are combined by a fixed tree.
__global__ void __launch_bounds__(256) finalize_norm_many_kernel(const float* partials, int npart, float eps,
                                                                 float* inv) {
  __shared__ double ws[8];
  const int b = blockIdx.x;
  const int per = (npart + 255) / 256;
  const int p0 = threadIdx.x * per;
  double s = 0.0;
  for (int p = p0; p < p0 + per && p < npart; ++p) s += (double)partials[(long long)b * npart + p];
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  if ((threadIdx.x & 31) == 0) ws[threadIdx.x >> 5] = s;
  __syncthreads();
  if (threadIdx.x == 0) {
    double t = 0.0;
    for (int w = 0; w < 8; ++w) t += ws[w];
    inv[b] = (float)(1.0 / (sqrt(t) + (double)eps));
  }
}

// inv[b] = 1 / (sqrt(sum of partials) + eps), partials summed in order in fp64.
__global__ void finalize_norm_kernel(const float* partials, int npart, int count, float eps, float* inv) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= count) return;
  double s = 0.0;
  for (int p = 0; p < npart; ++p) s += (double)partials[(long long)b * npart + p];
  inv[b] = (float)(1.0 / (sqrt(s) + (double)eps));
}

// ---------------------------------------------------------------------------------------
// exact l1 keys. A finite bf16 value with exponent field E and fraction f has magnitude
// mant * 2^(e-1) units of 2^-133, mant = (E ? 128 + f : f), e = max(E, 1). The key is the
// exact sum, kept as KEY_DIGITS base-2^32 digits; a thread accumulates digit sums in
// 64-bit registers (digit d = (e-1) >> 5 receives mant << ((e-1) & 31)) and carries them
// into canonical 32-bit digits before adding them into the row's key with integer atomics
// (order-independent). Rows with an Inf/NaN are flagged in nf.

struct KeyAcc {
  uint64_t acc[8];
  uint64_t cur;
  uint32_t dcur;
  bool nonfinite;
  __device__ void init() {
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0;
    cur = 0;
    dcur = 0;
    nonfinite = false;
  }
  __device__ __forceinline__ void flush() {
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if (dcur == (uint32_t)i) acc[i] += cur;
    cur = 0;
  }
  __device__ __forceinline__ void add(uint16_t bits) {
    const uint32_t E = (bits >> 7) & 0xFFu;
    if (E == 0xFFu) {
      nonfinite = true;
      return;
    }
    const uint32_t f = bits & 0x7Fu;
    const uint32_t mant = E ? (f | 0x80u) : f;
    if (!mant) return;
    const uint32_t ee = E ? E - 1u : 0u;
    const uint32_t d = ee >> 5;
    const uint64_t v = static_cast<uint64_t>(mant) << (ee & 31u);
    if (d != dcur) {
      flush();
      dcur = d;
    }
    cur += v;
  }
  // canonical digits (each < 2^32) of this thread's partial sum
  __device__ void digits(uint32_t (&dg)[KEY_DIGITS]) {
    flush();
    uint64_t carry = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint64_t t = acc[i] + carry;
      dg[i] = static_cast<uint32_t>(t);
      carry = t >> 32;
    }
    dg[8] = static_cast<uint32_t>(carry);
    dg[9] = static_cast<uint32_t>(carry >> 32);
  }
};

// The row kernel's accumulator: the same exact sum, counted in units of 2^-135 (every key
// of a matrix is four times the sum above, which leaves their order unchanged), with the
// eight digit sums in shared memory (one slot of 8 per thread; they change only when a
// value's exponent leaves the current digit, so keeping them out of registers costs little
// and lets more warps stream the matrix). With q = E - min(E, 1) + 2 a finite value adds
// mant << (q & 31) to digit q >> 5 (at most 7); Inf / NaN (E = 255) land in digit 8, which
// no finite value reaches, so they are caught on the rare path that changes digits, and
// zeros keep the current digit (they add nothing).
struct KeyAccS {
  uint64_t* acc;
  uint64_t cur;
  uint32_t dcur;
  bool nonfinite;
  __device__ void init(uint64_t* slot) {
    acc = slot;
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0;
    cur = 0;
    dcur = 0;
    nonfinite = false;
  }
  __device__ __forceinline__ void flush() {
    acc[dcur] += cur;
    cur = 0;
  }
  // one value given by its exponent field E and fraction f
  __device__ __forceinline__ void add(uint32_t E, uint32_t f) {
    const uint32_t h = min(E, 1u);
    const uint32_t mant = f + (h << 7);
    const uint32_t q = E - h + 2u;
    const uint32_t d = mant ? (q >> 5) : dcur;
    if (d != dcur) {
      if (d > 7u) {
        nonfinite = true;  // the row's key is replaced; what this lane adds no longer matters
      } else {
        flush();
        dcur = d;
      }
    }
    uint32_t lo, hi;  // mant << (q & 31) as a 64-bit value
    asm("shf.l.wrap.b32 %0, %1, %2, %3;" : "=r"(lo) : "r"(0u), "r"(mant), "r"(q));
    asm("shf.l.wrap.b32 %0, %1, %2, %3;" : "=r"(hi) : "r"(mant), "r"(0u), "r"(q));
    cur += (static_cast<uint64_t>(hi) << 32) | lo;
  }
  // both bf16 values of a 32-bit word
  __device__ __forceinline__ void add2(uint32_t w) {
    add((w >> 7) & 0xFFu, w & 0x7Fu);
    add((w >> 23) & 0xFFu, (w >> 16) & 0x7Fu);
  }
  __device__ void digits(uint32_t (&dg)[KEY_DIGITS]) {
    flush();
    uint64_t carry = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint64_t t = acc[i] + carry;
      dg[i] = static_cast<uint32_t>(t);
      carry = t >> 32;
    }
    dg[8] = static_cast<uint32_t>(carry);
    dg[9] = static_cast<uint32_t>(carry >> 32);
  }
};

// M + G of two bf16 pairs, each sum rounded once to bf16 (a correctly rounded bf16 add is
// the fp32 sum rounded to bf16: fp32 holds more than twice bf16's significand bits, so the
// double rounding cannot differ)
__device__ __forceinline__ uint32_t bf16x2_add(uint32_t a, uint32_t b) {
  const __nv_bfloat162 r = __hadd2(*reinterpret_cast<const __nv_bfloat162*>(&a), *reinterpret_cast<const __nv_bfloat162*>(&b));
  return *reinterpret_cast<const uint32_t*>(&r);
}

// Rows of the (non-transposed) matrix: M <- M + G and the key of each row. One warp per
// row; per-lane digits are summed across the warp (each sum < 2^37) and stored.
__global__ void frac_add_keys_rows_kernel(bf16* M, long long ldm, long long sm, const bf16* G, long long ldg,
                                          long long sg, int rows, int cols, int count, unsigned long long* keys,
                                          int* nf) {
  const int warps_per_block = blockDim.x >> 5;
  const long long gw = (long long)blockIdx.x * warps_per_block + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (gw >= (long long)rows * count) return;
  const int b = (int)(gw / rows), r = (int)(gw % rows);
  bf16* mr = M + (long long)b * sm + (long long)r * ldm;
  const bf16* gr = G + (long long)b * sg + (long long)r * ldg;
  __shared__ uint64_t slots[256 * 8];
  KeyAccS ka;
  ka.init(slots + threadIdx.x * 8);
  const int cvec = cols & ~7;
  // software-pipelined: the next 16-byte vectors are in flight while this one is summed
  int c = lane * 8;
  uint4 mv = make_uint4(0, 0, 0, 0), gv = mv;
  if (c < cvec) {
    mv = *reinterpret_cast<const uint4*>(mr + c);
    gv = *reinterpret_cast<const uint4*>(gr + c);
  }
  for (; c < cvec; c += 32 * 8) {
    const int cn = c + 32 * 8;
    uint4 mn = make_uint4(0, 0, 0, 0), gn = mn;
    if (cn < cvec) {
      mn = *reinterpret_cast<const uint4*>(mr + cn);
      gn = *reinterpret_cast<const uint4*>(gr + cn);
    }
    mv.x = bf16x2_add(mv.x, gv.x);
    mv.y = bf16x2_add(mv.y, gv.y);
    mv.z = bf16x2_add(mv.z, gv.z);
    mv.w = bf16x2_add(mv.w, gv.w);
    *reinterpret_cast<uint4*>(mr + c) = mv;
    ka.add2(mv.x);
    ka.add2(mv.y);
    ka.add2(mv.z);
    ka.add2(mv.w);
    mv = mn;
    gv = gn;
  }
  for (int c = cvec + lane; c < cols; c += 32) {
    const bf16 nv = f_to_bf16(__fadd_rn(bf16_to_f(mr[c]), bf16_to_f(gr[c])));
    mr[c] = nv;
    const uint32_t u = __bfloat16_as_ushort(nv);
    ka.add((u >> 7) & 0xFFu, u & 0x7Fu);
  }
  uint32_t dg[KEY_DIGITS];
  ka.digits(dg);
  unsigned long long* kr = keys + ((long long)b * rows + r) * KEY_DIGITS;
  const unsigned any_nf = __any_sync(0xffffffffu, ka.nonfinite);
#pragma unroll
  for (int i = 0; i < KEY_DIGITS; ++i) {
    unsigned long long s = dg[i];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (lane == 0) kr[i] = s;
  }
  if (lane == 0) nf[(long long)b * rows + r] = any_nf ? 1 : 0;
}

// Columns of the matrix (rows of its transpose): M <- M + G elementwise and the key of
// every column, one thread per column over a chunk of rows, digits added with atomics.
// keys / nf must be zero on entry.
__global__ void frac_add_keys_cols_kernel(bf16* M, long long ldm, long long sm, const bf16* G, long long ldg,
                                          long long sg, int rows, int cols, int rows_per_chunk,
                                          unsigned long long* keys, int* nf) {
  const int b = blockIdx.z;
  const int c = blockIdx.x * blockDim.x + threadIdx.x;
  if (c >= cols) return;
  const int r0 = blockIdx.y * rows_per_chunk, r1 = min(rows, r0 + rows_per_chunk);
  bf16* Mb = M + (long long)b * sm;
  const bf16* Gb = G + (long long)b * sg;
  KeyAcc ka;
  ka.init();
  for (int r = r0; r < r1; ++r) {
    const bf16 nv = f_to_bf16(__fadd_rn(bf16_to_f(Mb[(long long)r * ldm + c]), bf16_to_f(Gb[(long long)r * ldg + c])));
    Mb[(long long)r * ldm + c] = nv;
    ka.add(__bfloat16_as_ushort(nv));
  }
  uint32_t dg[KEY_DIGITS];
  ka.digits(dg);
  unsigned long long* kc = keys + ((long long)b * cols + c) * KEY_DIGITS;
#pragma unroll
  for (int i = 0; i < KEY_DIGITS; ++i)
    if (dg[i]) atomicAdd(kc + i, (unsigned long long)dg[i]);
  if (ka.nonfinite) atomicOr(nf + (long long)b * cols + c, 1);
}

// Columns of the matrix, 16-byte vectors: the same pass with each thread on 8 adjacent
// columns (one vector of M and of G per row) over a chunk of rows, M + G by packed bf16x2
// adds. Every column keeps, in registers, the running sum of its current digit window in
// the row kernel's units (2^-135, digit window q >> 5 with q = E - min(E, 1) + 2; keys of
// one matrix all come from this kernel, so only their order matters); a window change, and
// the end of the chunk, add that sum into the column's key digit with a 64-bit atomic
// (integer sums: order-independent), to be carried into canonical digits by the selection
// kernel. Inf / NaN land in window 8 and flag the column. keys / nf must be zero on entry;
// cols must be a multiple of 8 and the rows 16-byte aligned.
struct ColKeys8 {
  uint64_t cur[8];
  uint32_t dcur[8];
  uint32_t nonfinite;  // bit e: column e saw an Inf / NaN
  __device__ __forceinline__ void init() {
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      cur[e] = 0;
      dcur[e] = 0;
    }
    nonfinite = 0;
  }
  // Columns e and e + 1 from one word of two bf16 values (e in the low half): the exponent and
  // mantissa fields of both are formed with 32-bit operations on the pair
  // (no carry or borrow crosses the halves: mant <= 255, q <= 256, E >= min(E, 1)).
  __device__ __forceinline__ void add2(int e, uint32_t w, unsigned long long* key) {
    const uint32_t E2 = (w >> 7) & 0x00FF00FFu;
    const uint32_t h2 = ((E2 + 0x00FF00FFu) >> 8) & 0x00010001u;  // min(E, 1): E + 255 reaches bit 8 iff E > 0
    const uint32_t mant2 = (w & 0x007F007Fu) + (h2 << 7);
    const uint32_t q2 = E2 - h2 + 0x00020002u;
    step(e, mant2 & 0xFFFFu, q2 & 0xFFFFu, key);
    step(e + 1, mant2 >> 16, q2 >> 16, key + KEY_DIGITS);
  }
  // One value of column e: a change of digit window adds the finished window sum into the
  // key; window 8 (Inf / NaN) flags the column, whose key is then replaced.
  __device__ __forceinline__ void step(int e, uint32_t mant, uint32_t q, unsigned long long* key) {
    const uint32_t d = mant ? (q >> 5) : dcur[e];
    if (d != dcur[e]) {
      if (d > 7u) {
        nonfinite |= 1u << e;
      } else {
        if (cur[e]) atomicAdd(key + dcur[e], (unsigned long long)cur[e]);
        cur[e] = 0;
        dcur[e] = d;
      }
    }
    uint32_t lo, hi;
    asm("shf.l.wrap.b32 %0, %1, %2, %3;" : "=r"(lo) : "r"(0u), "r"(mant), "r"(q));
    asm("shf.l.wrap.b32 %0, %1, %2, %3;" : "=r"(hi) : "r"(mant), "r"(0u), "r"(q));
    cur[e] += (static_cast<uint64_t>(hi) << 32) | lo;
  }
};

__global__ void __launch_bounds__(256) frac_add_keys_cols8_kernel(bf16* M, long long ldm, long long sm,
                                                                  const bf16* G, long long ldg, long long sg,
                                                                  int rows, int cols, int rows_per_chunk,
                                                                  unsigned long long* keys, int* nf) {
  const int b = blockIdx.z;
  const int c0 = (blockIdx.x * blockDim.x + threadIdx.x) * 8;
  if (c0 >= cols) return;
  const int r0 = blockIdx.y * rows_per_chunk, r1 = min(rows, r0 + rows_per_chunk);
  bf16* Mb = M + (long long)b * sm + c0;
  const bf16* Gb = G + (long long)b * sg + c0;
  unsigned long long* kb = keys + ((long long)b * cols + c0) * KEY_DIGITS;
  ColKeys8 ka;
  ka.init();
  uint4 mv = make_uint4(0, 0, 0, 0), gv = mv;
  if (r0 < r1) {
    mv = *reinterpret_cast<const uint4*>(Mb + (long long)r0 * ldm);
    gv = *reinterpret_cast<const uint4*>(Gb + (long long)r0 * ldg);
  }
  for (int r = r0; r < r1; ++r) {
    // the next row's vectors are in flight while this one is summed
    uint4 mn = make_uint4(0, 0, 0, 0), gn = mn;
    if (r + 1 < r1) {
      mn = *reinterpret_cast<const uint4*>(Mb + (long long)(r + 1) * ldm);
      gn = *reinterpret_cast<const uint4*>(Gb + (long long)(r + 1) * ldg);
    }
    mv.x = bf16x2_add(mv.x, gv.x);
    mv.y = bf16x2_add(mv.y, gv.y);
    mv.z = bf16x2_add(mv.z, gv.z);
    mv.w = bf16x2_add(mv.w, gv.w);
    *reinterpret_cast<uint4*>(Mb + (long long)r * ldm) = mv;
    const uint32_t w[4] = {mv.x, mv.y, mv.z, mv.w};
#pragma unroll
    for (int e = 0; e < 8; e += 2) ka.add2(e, w[e >> 1], kb + (long long)e * KEY_DIGITS);
    mv = mn;
    gv = gn;
  }
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    if (ka.cur[e]) atomicAdd(kb + (long long)e * KEY_DIGITS + ka.dcur[e], (unsigned long long)ka.cur[e]);
    if ((ka.nonfinite >> e) & 1u) atomicOr(nf + (long long)b * cols + c0 + e, 1);
  }
}

// Keys of the rows (trans = 0) or columns (trans = 1) of M, without updating M.
__global__ void keys_only_kernel(const bf16* M, long long ldm, long long sm, int rows, int cols, int trans,
                                 int rows_per_chunk, unsigned long long* keys, int* nf) {
  const int b = blockIdx.z;
  const bf16* Mb = M + (long long)b * sm;
  KeyAcc ka;
  ka.init();
  int key_index, nkeys;
  if (!trans) {
    // one thread per (row, column chunk): columns [c0, c1)
    const int r = blockIdx.y;
    const int c0 = (blockIdx.x * blockDim.x + threadIdx.x) * rows_per_chunk;
    if (c0 >= cols) return;
    const int c1 = min(cols, c0 + rows_per_chunk);
    for (int c = c0; c < c1; ++c) ka.add(__bfloat16_as_ushort(Mb[(long long)r * ldm + c]));
    key_index = r;
    nkeys = rows;
  } else {
    const int c = blockIdx.x * blockDim.x + threadIdx.x;
    if (c >= cols) return;
    const int r0 = blockIdx.y * rows_per_chunk, r1 = min(rows, r0 + rows_per_chunk);
    for (int r = r0; r < r1; ++r) ka.add(__bfloat16_as_ushort(Mb[(long long)r * ldm + c]));
    key_index = c;
    nkeys = cols;
  }
  uint32_t dg[KEY_DIGITS];
  ka.digits(dg);
  unsigned long long* kk = keys + ((long long)b * nkeys + key_index) * KEY_DIGITS;
#pragma unroll
  for (int i = 0; i < KEY_DIGITS; ++i)
    if (dg[i]) atomicAdd(kk + i, (unsigned long long)dg[i]);
  if (ka.nonfinite) atomicOr(nf + (long long)b * nkeys + key_index, 1);
}

// ---------------------------------------------------------------------------------------
// top-k selection per matrix (one block of 1024 threads each): exact radix select over
// the KEY_DIGITS*4 bytes of the keys from the most significant byte down; keys equal to
// the k-th largest go to the lowest indices; the k indices are written ascending.

__device__ int block_exclusive_scan_1024(int v, int* total) {
  __shared__ int wsum[32];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  __syncthreads();
  if (lane == 31) wsum[w] = x;
  __syncthreads();
  if (w == 0) {
    int s = wsum[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    wsum[lane] = s;  // inclusive
  }
  __syncthreads();
  const int base = w ? wsum[w - 1] : 0;
  *total = wsum[31];
  return base + x - v;
}

__global__ void __launch_bounds__(1024) select_topk_kernel(unsigned long long* keys, const int* nf, int n, int k,
                                                           int* idx) {
  extern __shared__ uint8_t st[];  // n states: 0 candidate, 1 selected, 2 rejected
  __shared__ unsigned hist[256];
  __shared__ int sh_T, sh_kleft, sh_cnt, sh_top;
  const int b = blockIdx.x;
  unsigned long long* K = keys + (long long)b * n * KEY_DIGITS;
  const int* F = nf + (long long)b * n;
  // canonicalise digits (carry propagation); non-finite rows get the key 2^319
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    unsigned long long* kr = K + (long long)i * KEY_DIGITS;
    if (F[i]) {
      for (int d = 0; d < KEY_DIGITS; ++d) kr[d] = 0;
      kr[KEY_DIGITS - 1] = 0x80000000ull;
    } else {
      unsigned long long carry = 0;
      for (int d = 0; d < KEY_DIGITS; ++d) {
        const unsigned long long t = kr[d] + carry;
        kr[d] = t & 0xFFFFFFFFull;
        carry = t >> 32;
      }
    }
    st[i] = 0;
  }
  if (threadIdx.x == 0) sh_top = 0;
  __syncthreads();
  // the most significant non-zero key byte: the bytes above it are zero in every key, so
  // the radix passes start there
  {
    int top = 0;
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
      const unsigned long long* kr = K + (long long)i * KEY_DIGITS;
      for (int d = KEY_DIGITS - 1; d >= 0; --d)
        if (kr[d]) {
          top = max(top, d * 4 + (31 - __clz((unsigned)kr[d])) / 8);
          break;
        }
    }
    atomicMax(&sh_top, top);
  }
  int kleft = k;
  __syncthreads();
  for (int p = sh_top; p >= 0; --p) {
    for (int h = threadIdx.x; h < 256; h += blockDim.x) hist[h] = 0;
    __syncthreads();
    const int dg = p >> 2, sh = (p & 3) * 8;
    for (int i = threadIdx.x; i < n; i += blockDim.x)
      if (st[i] == 0) atomicAdd(&hist[(K[(long long)i * KEY_DIGITS + dg] >> sh) & 0xFF], 1u);
    __syncthreads();
    if (threadIdx.x < 32) {
      // the bucket T holding the kleft-th largest candidate, found by warp 0: lane l sums
      // buckets 255 - 8l down to 248 - 8l, a warp scan gives the counts above each lane's
      // group, and the lane whose group crosses kleft walks its eight buckets
      const int lane = threadIdx.x;
      int grp = 0;
#pragma unroll
      for (int e = 0; e < 8; ++e) grp += (int)hist[255 - 8 * lane - e];
      int incl = grp;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      const int above = incl - grp;  // candidates in the buckets above this lane's group
      const unsigned hit = __ballot_sync(0xffffffffu, above < kleft && incl >= kleft);
      if (lane == __ffs(hit) - 1) {
        int cum = above, T = 255 - 8 * lane;
        for (int e = 0; e < 8; ++e) {
          const int bk = 255 - 8 * lane - e;
          if (cum + (int)hist[bk] >= kleft) {
            T = bk;
            break;
          }
          cum += (int)hist[bk];
        }
        sh_T = T;
        sh_kleft = kleft - cum;
        sh_cnt = (int)hist[T];
      }
    }
    __syncthreads();
    const unsigned T = (unsigned)sh_T;
    for (int i = threadIdx.x; i < n; i += blockDim.x)
      if (st[i] == 0) {
        const unsigned by = (unsigned)((K[(long long)i * KEY_DIGITS + dg] >> sh) & 0xFF);
        st[i] = by > T ? 1 : (by < T ? 2 : 0);
      }
    kleft = sh_kleft;
    const int cnt = sh_cnt;
    __syncthreads();
    if (cnt == kleft) break;  // every remaining candidate is selected
  }
  // remaining candidates hold equal keys: the kleft lowest indices are selected
  const int seg = (n + blockDim.x - 1) / blockDim.x;
  const int i0 = min(n, (int)threadIdx.x * seg), i1 = min(n, i0 + seg);
  int c = 0;
  for (int i = i0; i < i1; ++i) c += st[i] == 0;
  int tot;
  int rank = block_exclusive_scan_1024(c, &tot);
  for (int i = i0; i < i1; ++i)
    if (st[i] == 0) {
      st[i] = rank < kleft ? 1 : 2;
      ++rank;
    }
  __syncthreads();
  c = 0;
  for (int i = i0; i < i1; ++i) c += st[i] == 1;
  int pos = block_exclusive_scan_1024(c, &tot);
  int* out = idx + (long long)b * k;
  for (int i = i0; i < i1; ++i)
    if (st[i] == 1) {
      if (pos < k) out[pos] = i;
      ++pos;
    }
}

// ---------------------------------------------------------------------------------------
// gathers, decays, copies

// X[b][i][:] = M[b][idx[b*k + i]][:] (rows), with sum-of-squares partials of X.
// With decay, the selected rows of M are also replaced by bf16(mu * M) (Dion3 Algorithm 4's
// error feedback) once copied: nothing reads M[S] after the gather, so the decay
// rides on this pass.
__global__ void gather_rows_kernel(bf16* M, long long ldm, long long sm, const int* idx, int k, int cols,
                                   bf16* X, long long ldx, long long sx, int npart, float* partials, int decay,
                                   float mu) {
  const int b = blockIdx.y, part = blockIdx.x;
  const int rp = (k + npart - 1) / npart;
  const int i0 = part * rp, i1 = min(k, i0 + rp);
  float acc = 0.f;
  for (int i = i0; i < i1; ++i) {
    const int r = idx[(long long)b * k + i];
    bf16* src = M + (long long)b * sm + (long long)r * ldm;
    bf16* dst = X + (long long)b * sx + (long long)i * ldx;
    const int cvec = cols & ~7;
    // GV vectors of the row per thread are loaded before the first store (a store to M or X
    // may alias the next load as far as the compiler knows, so a load after it would wait)
    constexpr int GV = 8;
    for (int c0 = threadIdx.x * 8; c0 < cvec; c0 += GV * blockDim.x * 8) {
      uint4 u[GV];
#pragma unroll
      for (int j = 0; j < GV; ++j) {
        const int c = c0 + j * blockDim.x * 8;
        u[j] = c < cvec ? *reinterpret_cast<const uint4*>(src + c) : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int j = 0; j < GV; ++j) {
        const int c = c0 + j * blockDim.x * 8;
        if (c >= cvec) break;
        *reinterpret_cast<uint4*>(dst + c) = u[j];
        const bf16* e = reinterpret_cast<const bf16*>(&u[j]);
        uint4 dv;
        bf16* de = reinterpret_cast<bf16*>(&dv);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const float f = bf16_to_f(e[q]);
          acc = fmaf(f, f, acc);
          de[q] = f_to_bf16(__fmul_rn(mu, f));
        }
        if (decay) *reinterpret_cast<uint4*>(src + c) = dv;
      }
    }
    for (int c = cvec + threadIdx.x; c < cols; c += blockDim.x) {
      const bf16 v = src[c];
      dst[c] = v;
      const float f = bf16_to_f(v);
      acc = fmaf(f, f, acc);
      if (decay) src[c] = f_to_bf16(__fmul_rn(mu, f));
    }
  }
  const float s = block_sum_256(acc);
  if (threadIdx.x == 0) partials[(long long)b * npart + part] = s;
}

// Rows per block of the column gather / scatter of a tall matrix (32 selected columns wide).
constexpr int COL_TILE_ROWS = 64;

// X[b][i][j] = M[b][j][idx[b*k + i]] (columns of M become rows of X), with the decay
// M[b][j][idx[i]] = bf16(mu * M) when asked; 32 x TJ tiles staged in shared memory. With
// bpart, each block also stores the sum of squares of the values it gathered, in a fixed
// order (per thread, then the fixed block tree), at bpart[b * blocks + its index].
template <int TJ>
__global__ void __launch_bounds__(256) gather_cols_kernel(bf16* M, long long ldm, long long sm, const int* idx, int k,
                                                          int rows, bf16* X, long long ldx, long long sx, int decay,
                                                          float mu, float* bpart) {
  // 32 selected columns x TJ rows per block: each thread issues its TJ / 8 loads before
  // using any of them
  __shared__ bf16 tile[TJ][33];
  constexpr int R = TJ / 8;
  const int b = blockIdx.z;
  const int i0 = blockIdx.x * 32, j0 = blockIdx.y * TJ;
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;  // 32 x 8
  const int i = i0 + tx;
  const bool iv = i < k;
  bf16* col = M + (long long)b * sm + (iv ? idx[(long long)b * k + i] : 0);
  bf16 v[R];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const int j = j0 + ty + 8 * r;
    v[r] = f_to_bf16(0.f);
    if (iv && j < rows) v[r] = col[(long long)j * ldm];
  }
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const int j = j0 + ty + 8 * r;
    if (decay && iv && j < rows) col[(long long)j * ldm] = f_to_bf16(__fmul_rn(mu, bf16_to_f(v[r])));
    tile[ty + 8 * r][tx] = v[r];
  }
  if (bpart) {
    float q = 0.f;
#pragma unroll
    for (int r = 0; r < R; ++r) q = fmaf(bf16_to_f(v[r]), bf16_to_f(v[r]), q);
    q = block_sum_256(q);
    if (threadIdx.x == 0)
      bpart[(long long)b * gridDim.x * gridDim.y + (long long)blockIdx.y * gridDim.x + blockIdx.x] = q;
  }
  __syncthreads();
  for (int ii = ty; ii < 32; ii += 8) {
    const int iw = i0 + ii;
    if (iw >= k) break;
#pragma unroll
    for (int jj = tx; jj < TJ; jj += 32) {
      const int j = j0 + jj;
      if (j < rows) X[(long long)b * sx + (long long)iw * ldx + j] = tile[jj][ii];
    }
  }
}

// flags[b*n + idx[b*k + i]] = 1 (flags zeroed before).
__global__ void mark_selected_kernel(const int* idx, int k, int n, int count, int* flags) {
  const long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= (long long)k * count) return;
  const int b = (int)(e / k);
  flags[(long long)b * n + idx[e]] = 1;
}

// Rows (trans = 0) or columns (trans = 1) of W whose flag is 0 get W <- bf16(factor W); a
// block per ROWS_PER_BLOCK rows, 16-byte vectors.
__global__ void scale_unselected_kernel(bf16* W, long long ldw, long long sw, int rows, int cols, const int* flags,
                                        int trans, float factor) {
  const int b = blockIdx.y;
  const int nf = trans ? cols : rows;
  const int* F = flags + (long long)b * nf;
  const int cvec = cols & ~7;
  for (int r = blockIdx.x * ROWS_PER_BLOCK; r < min(rows, (int)(blockIdx.x + 1) * ROWS_PER_BLOCK); ++r) {
    if (!trans && F[r]) continue;
    bf16* row = W + (long long)b * sw + (long long)r * ldw;
    for (int c = threadIdx.x * 8; c < cvec; c += blockDim.x * 8) {
      uint4 u = *reinterpret_cast<const uint4*>(row + c);
      bf16* e = reinterpret_cast<bf16*>(&u);
#pragma unroll
      for (int q = 0; q < 8; ++q)
        if (!trans || !F[c + q]) e[q] = f_to_bf16(__fmul_rn(factor, bf16_to_f(e[q])));
      *reinterpret_cast<uint4*>(row + c) = u;
    }
    for (int c = cvec + threadIdx.x; c < cols; c += blockDim.x)
      if (!trans || !F[c]) row[c] = f_to_bf16(__fmul_rn(factor, bf16_to_f(row[c])));
  }
}

// Selected rows of W take beta * W + alpha * r_i * O: W[idx[i]][j] for O[i][j], i < k,
// j < len; fp32 arithmetic, one rounding (the weight update of Dion3 sec. 6 on the selected
// rows only). idx == NULL selects every row (i itself); rs == NULL means r_i = 1 (NorMuon
// passes its row scales). One block per row of O, 16-byte vectors.
__global__ void scatter_update_rows_kernel(bf16* W, long long ldw, long long sw, const bf16* O, long long ldo,
                                           long long so, const int* idx, const float* rs, int k, int len, float alpha,
                                           float beta) {
  const int b = blockIdx.y, i = blockIdx.x;
  const long long e = (long long)b * k + i;
  const int sel = idx ? idx[e] : i;
  const float a = rs ? alpha * rs[e] : alpha;
  bf16* wr = W + (long long)b * sw + (long long)sel * ldw;
  const bf16* orow = O + (long long)b * so + (long long)i * ldo;
  const int cvec = len & ~7;
  for (int c = threadIdx.x * 8; c < cvec; c += blockDim.x * 8) {
    uint4 wu = *reinterpret_cast<const uint4*>(wr + c);
    const uint4 ou = *reinterpret_cast<const uint4*>(orow + c);
    bf16* we = reinterpret_cast<bf16*>(&wu);
    const bf16* oe = reinterpret_cast<const bf16*>(&ou);
#pragma unroll
    for (int q = 0; q < 8; ++q) we[q] = f_to_bf16(fmaf(a, bf16_to_f(oe[q]), beta * bf16_to_f(we[q])));
    *reinterpret_cast<uint4*>(wr + c) = wu;
  }
  for (int c = cvec + threadIdx.x; c < len; c += blockDim.x)
    wr[c] = f_to_bf16(fmaf(a, bf16_to_f(orow[c]), beta * bf16_to_f(wr[c])));
}

// The same for the columns of a tall W: W[j][idx[i]] for O[i][j]. A 32 x TJ tile of O goes
// through shared memory so that both the O reads and the W accesses are along rows.
template <int TJ>
__global__ void __launch_bounds__(256) scatter_update_cols_kernel(bf16* W, long long ldw, long long sw, const bf16* O,
                                                                  long long ldo, long long so, const int* idx,
                                                                  const float* rs, int k, int len, float alpha,
                                                                  float beta) {
  // 32 selected columns x TJ rows per block; the TJ / 8 loads of W a thread makes are all
  // issued before the first update
  __shared__ float tile[32][TJ + 1];
  constexpr int R = TJ / 8;
  const int b = blockIdx.z;
  const int i0 = blockIdx.x * 32, j0 = blockIdx.y * TJ;
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;  // 32 x 8
  for (int ii = ty; ii < 32; ii += 8) {
    const int i = i0 + ii;
#pragma unroll
    for (int jj = tx; jj < TJ; jj += 32) {
      const int j = j0 + jj;
      float v = 0.f;
      if (i < k && j < len) {
        v = bf16_to_f(O[(long long)b * so + (long long)i * ldo + j]);
        if (rs) v *= rs[(long long)b * k + i];
      }
      tile[ii][jj] = v;
    }
  }
  __syncthreads();
  const int i = i0 + tx;
  if (i >= k) return;
  bf16* col = W + (long long)b * sw + (idx ? idx[(long long)b * k + i] : i);
  bf16 w[R];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const int j = j0 + ty + 8 * r;
    if (j < len) w[r] = col[(long long)j * ldw];
  }
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const int j = j0 + ty + 8 * r;
    if (j < len) col[(long long)j * ldw] = f_to_bf16(fmaf(alpha, tile[tx][ty + 8 * r], beta * bf16_to_f(w[r])));
  }
}

// The same update from the transpose of O (OT[j][i] = O[i][j], len x k): W[j][idx[i]] =
// bf16(beta W + alpha OT[j][i]). A block covers 32 selected columns x TJ rows; a warp reads
// 32 consecutive entries of an OT row and the 32 selected entries of the same W row, and
// each thread issues all its loads of W and OT before its first update.
template <int TJ>
__global__ void __launch_bounds__(256) scatter_update_cols_t_kernel(bf16* W, long long ldw, long long sw,
                                                                    const bf16* OT, long long ldo, long long so,
                                                                    const int* idx, int k, int len, float alpha,
                                                                    float beta) {
  constexpr int R = TJ / 8;
  const int b = blockIdx.z;
  const int i = blockIdx.x * 32 + (threadIdx.x & 31);
  const int j0 = blockIdx.y * TJ + (threadIdx.x >> 5);
  if (i >= k) return;
  bf16* col = W + (long long)b * sw + idx[(long long)b * k + i];
  const bf16* oc = OT + (long long)b * so + i;
  bf16 w[R], o[R];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const int j = j0 + 8 * r;
    if (j < len) {
      w[r] = col[(long long)j * ldw];
      o[r] = oc[(long long)j * ldo];
    }
  }
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const int j = j0 + 8 * r;
    if (j < len) col[(long long)j * ldw] = f_to_bf16(fmaf(alpha, bf16_to_f(o[r]), beta * bf16_to_f(w[r])));
  }
}

// ---------------------------------------------------------------------------------------
// NorMuon and RowNorm statistics

// s[b*k + i] = sum_j X[b][i][j]^2 over the k rows of X (bf16), one warp per row, lanes on
// 16-byte vectors in a fixed order.
__global__ void row_sumsq_kernel(const bf16* X, long long ldx, long long sx, int k, int cols, int count, float* s) {
  const long long row = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= (long long)k * count) return;
  const int b = (int)(row / k), i = (int)(row % k);
  const bf16* r = X + (long long)b * sx + (long long)i * ldx;
  float acc = 0.f;
  const int cvec = cols & ~7;
#pragma unroll 4
  for (int c = lane * 8; c < cvec; c += 32 * 8) {
    const uint4 u = *reinterpret_cast<const uint4*>(r + c);
    const bf16* e = reinterpret_cast<const bf16*>(&u);
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const float v = bf16_to_f(e[q]);
      acc = fmaf(v, v, acc);
    }
  }
  for (int c = cvec + lane; c < cols; c += 32) {
    const float v = bf16_to_f(r[c]);
    acc = fmaf(v, v, acc);
  }
  acc = warp_sum(acc);
  if (lane == 0) s[row] = acc;
}

// Column sums of squares of M (rows x cols, bf16) in NPART row slices:
// part[(b * NPART + p) * cols + c]; a thread owns one column of one slice.
__global__ void col_sumsq_part_kernel(const bf16* M, long long ldm, long long sm, int rows, int cols, int npart,
                                      float* part) {
  const int b = blockIdx.z, p = blockIdx.y;
  const int c = blockIdx.x * blockDim.x + threadIdx.x;
  if (c >= cols) return;
  const int rp = (rows + npart - 1) / npart;
  const int r0 = p * rp, r1 = min(rows, r0 + rp);
  const bf16* Mb = M + (long long)b * sm;
  float acc = 0.f;
  for (int r = r0; r < r1; ++r) {
    const float v = bf16_to_f(Mb[(long long)r * ldm + c]);
    acc = fmaf(v, v, acc);
  }
  part[((long long)b * npart + p) * cols + c] = acc;
}

// s[b*cols + c] = sum of the NPART slice sums, in slice order.
__global__ void col_sumsq_finish_kernel(const float* part, int cols, int npart, int count, float* s) {
  const long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= (long long)cols * count) return;
  const int b = (int)(e / cols), c = (int)(e % cols);
  float acc = 0.f;
  for (int p = 0; p < npart; ++p) acc += part[((long long)b * npart + p) * cols + c];
  s[e] = acc;
}

// NorMuon (Dion3 eq. (2); the NorMuon steps of Algorithm 4), one block per matrix. For the k rows of O
// with sums of squares s_i (of `len` columns each), row i being row sel(i) of the oriented
// matrix (sel = idx or the identity):
//   v <- beta2 v + (1 - beta2) s_i / len;  d_i = sqrt(v) + eps;
//   r_i = (||O||_F / ||O / d||_F) / d_i, the factor that turns O_ij into the rescaled
//   NorMuon update r_i O_ij.
// The norms are reduced in fp64 in a fixed order; the per-row quantities are fp32.
__global__ void __launch_bounds__(256) normuon_rows_kernel(const float* s, float* V, long long ldv, long long sv,
                                                           const int* idx, int k, int len, float beta2, float eps,
                                                           float* r) {
  __shared__ double red[2][256];
  const int b = blockIdx.x;
  double o2 = 0.0, h2 = 0.0;
  for (int i = threadIdx.x; i < k; i += blockDim.x) {
    const int sel = idx ? idx[(long long)b * k + i] : i;
    float* vp = V + (long long)b * sv + sel;
    const float si = s[(long long)b * k + i];
    const float v = fmaf(beta2, *vp, (1.f - beta2) * (si / (float)len));
    *vp = v;
    const float d = sqrtf(v) + eps;
    r[(long long)b * k + i] = d;
    o2 += (double)si;
    h2 += (double)si / ((double)d * (double)d);
  }
  red[0][threadIdx.x] = o2;
  red[1][threadIdx.x] = h2;
  __syncthreads();
  for (int w = blockDim.x / 2; w > 0; w >>= 1) {
    if (threadIdx.x < w) {
      red[0][threadIdx.x] += red[0][threadIdx.x + w];
      red[1][threadIdx.x] += red[1][threadIdx.x + w];
    }
    __syncthreads();
  }
  const double f = red[1][0] > 0.0 ? sqrt(red[0][0] / red[1][0]) : 0.0;
  for (int i = threadIdx.x; i < k; i += blockDim.x) {
    const long long e = (long long)b * k + i;
    r[e] = (float)(f / (double)r[e]);
  }
}

// One RowNorm step on the rows of a wide matrix in a single pass (Scaling Muon for DiTs
// eq. (5), (7) off a refresh step): per row, M <- bf16(mu M + G) (fp32 product, fp32 sum),
// s = sum of the stored M^2, r = gamma / max(sqrt(s), eps), W <- bf16(beta W + alpha r M).
// One block of 256 threads per row; the row's new M stays in registers (VPT 16-byte
// vectors per thread, cols = 2048 VPT at most, a multiple of 8): reads G, M, W and writes
// M, W once, the algorithmic minimum of 10 bytes per element.
template <int VPT>
__global__ void __launch_bounds__(256) rownorm_fused_rows_kernel(bf16* M, long long ldm, long long sm, const bf16* G,
                                                                 long long ldg, long long sg, bf16* W, long long ldw,
                                                                 long long sw, int cols, float mu, float gamma,
                                                                 float eps, float alpha, float beta) {
  const int b = blockIdx.y, i = blockIdx.x;
  bf16* mr = M + (long long)b * sm + (long long)i * ldm;
  const bf16* gr = G + (long long)b * sg + (long long)i * ldg;
  bf16* wr = W + (long long)b * sw + (long long)i * ldw;
  uint4 mv[VPT];
  float acc = 0.f;
#pragma unroll
  for (int v = 0; v < VPT; ++v) {
    const int c = (v * 256 + threadIdx.x) * 8;
    if (c < cols) {
      uint4 m4 = *reinterpret_cast<const uint4*>(mr + c);
      const uint4 g4 = *reinterpret_cast<const uint4*>(gr + c);
      bf16* me = reinterpret_cast<bf16*>(&m4);
      const bf16* ge = reinterpret_cast<const bf16*>(&g4);
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        me[q] = f_to_bf16(__fadd_rn(__fmul_rn(mu, bf16_to_f(me[q])), bf16_to_f(ge[q])));
        const float f = bf16_to_f(me[q]);
        acc = fmaf(f, f, acc);
      }
      *reinterpret_cast<uint4*>(mr + c) = m4;
      mv[v] = m4;
    }
  }
  __shared__ float r_sh;
  const float tot = block_sum_256(acc);
  if (threadIdx.x == 0) r_sh = gamma / fmaxf(sqrtf(tot), eps);
  __syncthreads();
  const float a = alpha * r_sh;
#pragma unroll
  for (int v = 0; v < VPT; ++v) {
    const int c = (v * 256 + threadIdx.x) * 8;
    if (c < cols) {
      uint4 w4 = *reinterpret_cast<const uint4*>(wr + c);
      bf16* we = reinterpret_cast<bf16*>(&w4);
      const bf16* me = reinterpret_cast<const bf16*>(&mv[v]);
#pragma unroll
      for (int q = 0; q < 8; ++q) we[q] = f_to_bf16(fmaf(a, bf16_to_f(me[q]), beta * bf16_to_f(we[q])));
      *reinterpret_cast<uint4*>(wr + c) = w4;
    }
  }
}

// RowNorm scales (Scaling Muon for DiTs eq. (5), multiplier gamma): r = gamma / max(sqrt(s), eps).
__global__ void rownorm_scale_kernel(const float* s, long long n, float gamma, float eps, float* r) {
  const long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= n) return;
  r[e] = gamma / fmaxf(sqrtf(s[e]), eps);
}

// W <- beta W + alpha r_q Y with q the row (trans = 0) or the column (trans = 1) of each
// element: a per-oriented-row scaled update, W and Y in the same physical layout. fp32
// arithmetic, one rounding; a block per ROWS_PER_BLOCK rows, 16-byte vectors.
__global__ void rowscale_update_kernel(bf16* W, long long ldw, long long sw, const bf16* Y, long long ldy,
                                       long long sy, const float* r, int rows, int cols, int trans, float alpha,
                                       float beta) {
  const int b = blockIdx.y;
  const float* R = r + (long long)b * (trans ? cols : rows);
  const int cvec = cols & ~7;
  for (int i = blockIdx.x * ROWS_PER_BLOCK; i < min(rows, (int)(blockIdx.x + 1) * ROWS_PER_BLOCK); ++i) {
    bf16* wr = W + (long long)b * sw + (long long)i * ldw;
    const bf16* yr = Y + (long long)b * sy + (long long)i * ldy;
    const float ar = trans ? alpha : alpha * R[i];
    for (int c = threadIdx.x * 8; c < cvec; c += blockDim.x * 8) {
      uint4 wu = *reinterpret_cast<const uint4*>(wr + c);
      const uint4 yu = *reinterpret_cast<const uint4*>(yr + c);
      bf16* we = reinterpret_cast<bf16*>(&wu);
      const bf16* ye = reinterpret_cast<const bf16*>(&yu);
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const float a = trans ? alpha * R[c + q] : ar;
        we[q] = f_to_bf16(fmaf(a, bf16_to_f(ye[q]), beta * bf16_to_f(we[q])));
      }
      *reinterpret_cast<uint4*>(wr + c) = wu;
    }
    for (int c = cvec + threadIdx.x; c < cols; c += blockDim.x) {
      const float a = trans ? alpha * R[c] : ar;
      wr[c] = f_to_bf16(fmaf(a, bf16_to_f(yr[c]), beta * bf16_to_f(wr[c])));
    }
  }
}

// X16 = fp16(inv[b] * M) in the same layout (Dion3 Algorithm 3's first steps for a bf16
// momentum: normalise, then round once to float16); 16-byte vectors.
__global__ void cast_scaled_kernel(__half* X, long long ldx, long long sx, const bf16* M, long long ldm, long long sm,
                                   const float* inv, int rows, int cols) {
  const int b = blockIdx.y;
  const float s = inv[b];
  const int cvec = cols & ~7;
  for (int i = blockIdx.x * ROWS_PER_BLOCK; i < min(rows, (int)(blockIdx.x + 1) * ROWS_PER_BLOCK); ++i) {
    const bf16* mr = M + (long long)b * sm + (long long)i * ldm;
    __half* xr = X + (long long)b * sx + (long long)i * ldx;
    for (int c = threadIdx.x * 8; c < cvec; c += blockDim.x * 8) {
      const uint4 mu = *reinterpret_cast<const uint4*>(mr + c);
      const bf16* me = reinterpret_cast<const bf16*>(&mu);
      uint4 xu;
      __half* xe = reinterpret_cast<__half*>(&xu);
#pragma unroll
      for (int q = 0; q < 8; ++q) xe[q] = __float2half_rn(s * bf16_to_f(me[q]));
      *reinterpret_cast<uint4*>(xr + c) = xu;
    }
    for (int c = cvec + threadIdx.x; c < cols; c += blockDim.x) xr[c] = __float2half_rn(s * bf16_to_f(mr[c]));
  }
}

// W <- beta * W + alpha * Y (same shape), fp32 arithmetic, one rounding.
template <typename TW, typename TY>
// (W and Y have elements of one size: 16-byte vectors of VEC elements along each row, a
// block per ROWS_PER_BLOCK rows.)
__global__ void axpby_kernel(TW* W, long long ldw, long long sw, const TY* Y, long long ldy, long long sy, int rows,
                             int cols, float alpha, float beta) {
  static_assert(sizeof(TW) == sizeof(TY), "W and Y share an element size");
  constexpr int VEC = 16 / sizeof(TW);
  const int b = blockIdx.y;
  const int cvec = cols - cols % VEC;
  for (int r = blockIdx.x * ROWS_PER_BLOCK; r < min(rows, (int)(blockIdx.x + 1) * ROWS_PER_BLOCK); ++r) {
    TW* wr = W + (long long)b * sw + (long long)r * ldw;
    const TY* yr = Y + (long long)b * sy + (long long)r * ldy;
    for (int c = threadIdx.x * VEC; c < cvec; c += blockDim.x * VEC) {
      uint4 wu = *reinterpret_cast<const uint4*>(wr + c);
      const uint4 yu = *reinterpret_cast<const uint4*>(yr + c);
      TW* we = reinterpret_cast<TW*>(&wu);
      const TY* ye = reinterpret_cast<const TY*>(&yu);
#pragma unroll
      for (int q = 0; q < VEC; ++q) we[q] = from_f<TW>(fmaf(alpha, to_f(ye[q]), beta * to_f(we[q])));
      *reinterpret_cast<uint4*>(wr + c) = wu;
    }
    for (int c = cvec + threadIdx.x; c < cols; c += blockDim.x)
      wr[c] = from_f<TW>(fmaf(alpha, to_f(yr[c]), beta * to_f(wr[c])));
  }
}

template <typename T>
__global__ void copy_kernel(T* D, long long ldd, long long sd, const T* S, long long lds, long long ss, int rows,
                            int cols) {
  const int b = blockIdx.z;
  const long long total = (long long)rows * cols;
  for (long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x; e < total; e += (long long)gridDim.x * blockDim.x) {
    const int r = (int)(e / cols), c = (int)(e % cols);
    D[(long long)b * sd + (long long)r * ldd + c] = S[(long long)b * ss + (long long)r * lds + c];
  }
}

// ---------------------------------------------------------------------------------------
// launchers

static cudaStream_t S(void* s) { return static_cast<cudaStream_t>(s); }

static int check_launch(const char* what, std::string* err) {
  profile_count_launch();
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    *err = std::string(what) + ": " + cudaGetErrorString(e);
    return GNS_ERR_CUDA;
  }
  return GNS_OK;
}

static unsigned grid_1d(long long work, int threads) {
  long long g = (work + threads - 1) / threads;
  const long long cap = (long long)device_sm_count() * 16;
  if (g > cap) g = cap;
  if (g < 1) g = 1;
  return (unsigned)g;
}

// ---------------------------------------------------------------------------------------
// failure detection without a fault: the bounded waits, made to run out

// One thread waits, through the same bounded-wait helpers the GEMM kernel uses for its
// cross-CTA completion counters and its mbarrier phases, first on *counter >= target and
// then on the first phase of an mbarrier that nothing arrives on, each for at most limit_ns.
// out[0] = nanoseconds spent in both waits, out[1] = bit 0 if the counter wait succeeded,
// bit 1 if the mbarrier wait did (it cannot). A wait that runs out sets GNS_DEVST_TIMEOUT.
__global__ void selftest_wait_kernel(const int* counter, int target, unsigned long long limit_ns, int* status,
                                     unsigned long long* out) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x != 0) return;
  mbar_init(&bar, 1);
  abort_flag = 0;
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  const uint64_t t0 = global_timer_ns();
  const bool c_ok = wait_counter(counter, target, &abort_flag, status, limit_ns);
  abort_flag = 0;  // the mbarrier wait then runs its own limit
  const bool m_ok = mbar_wait(&bar, 0u, &abort_flag, status, limit_ns);
  if (out) {
    out[0] = global_timer_ns() - t0;
    out[1] = (c_ok ? 1ull : 0ull) | (m_ok ? 2ull : 0ull);
  }
}

int launch_sumsq(gns_dtype dt, const MatRef& X, int64_t count, float* partials, void* stream, std::string* err,
                 int* zero, int nzero) {
  dim3 grid(NPART, (unsigned)count);
  if (dt == GNS_BF16)
    sumsq_kernel<bf16><<<grid, 256, 0, S(stream)>>>(static_cast<const bf16*>(X.ptr), X.ld, X.stride, (int)X.rows,
                                                   (int)X.cols, NPART, partials, zero, nzero);
  else if (dt == GNS_F16)
    sumsq_kernel<__half><<<grid, 256, 0, S(stream)>>>(static_cast<const __half*>(X.ptr), X.ld, X.stride, (int)X.rows,
                                                     (int)X.cols, NPART, partials, zero, nzero);
  else
    sumsq_kernel<float><<<grid, 256, 0, S(stream)>>>(static_cast<const float*>(X.ptr), X.ld, X.stride, (int)X.rows,
                                                    (int)X.cols, NPART, partials, zero, nzero);
  return check_launch("sumsq", err);
}

int launch_momentum(const MatRef& M, const MatRef& G, int64_t count, float mu, int mode, float* partials,
                    void* stream, std::string* err, int* zero, int nzero) {
  dim3 grid(NPART, (unsigned)count);
  momentum_kernel<<<grid, 256, 0, S(stream)>>>(static_cast<bf16*>(M.ptr), M.ld, M.stride,
                                               static_cast<const bf16*>(G.ptr), G.ld, G.stride, (int)M.rows,
                                               (int)M.cols, mu, mode, NPART, partials, zero, nzero);
  return check_launch("momentum", err);
}

int launch_finalize_norm(const float* partials, int64_t count, float eps, float* inv, void* stream, std::string* err,
                         int64_t npart) {
  if (npart <= NPART)
    finalize_norm_kernel<<<(unsigned)((count + 127) / 128), 128, 0, S(stream)>>>(partials, (int)npart, (int)count,
                                                                                  eps, inv);
  else
    finalize_norm_many_kernel<<<(unsigned)count, 256, 0, S(stream)>>>(partials, (int)npart, eps, inv);
  return check_launch("finalize_norm", err);
}

int64_t gather_cols_blocks(int64_t k, int64_t rows) {
  return ((k + 31) / 32) * ((rows + COL_TILE_ROWS - 1) / COL_TILE_ROWS);
}

int launch_frac_add_keys(const MatRef& M, const MatRef& G, int64_t count, int trans, unsigned long long* keys,
                         int* nf, void* stream, std::string* err) {
  if (!trans) {
    const long long rows_total = M.rows * count;
    const unsigned blocks = (unsigned)((rows_total + 7) / 8);
    frac_add_keys_rows_kernel<<<blocks, 256, 0, S(stream)>>>(static_cast<bf16*>(M.ptr), M.ld, M.stride,
                                                             static_cast<const bf16*>(G.ptr), G.ld, G.stride,
                                                             (int)M.rows, (int)M.cols, (int)count, keys, nf);
  } else {
    cudaMemsetAsync(keys, 0, sizeof(unsigned long long) * KEY_DIGITS * M.cols * count, S(stream));
    cudaMemsetAsync(nf, 0, sizeof(int) * M.cols * count, S(stream));
    const bool vec = M.cols % 8 == 0 && M.ld % 8 == 0 && G.ld % 8 == 0 && (count == 1 || (M.stride % 8 == 0 && G.stride % 8 == 0));
    if (vec) {
      // chunks of rows sized for about four waves of 8 resident blocks per SM
      const long long col_blocks = (M.cols / 8 + 255) / 256;
      const long long want = 4LL * 8 * device_sm_count();
      long long chunks = std::max(1LL, want / std::max(1LL, col_blocks * count));
      const int rpc = (int)std::max(64LL, (M.rows + chunks - 1) / chunks);
      dim3 grid((unsigned)col_blocks, (unsigned)((M.rows + rpc - 1) / rpc), (unsigned)count);
      frac_add_keys_cols8_kernel<<<grid, 256, 0, S(stream)>>>(static_cast<bf16*>(M.ptr), M.ld, M.stride,
                                                              static_cast<const bf16*>(G.ptr), G.ld, G.stride,
                                                              (int)M.rows, (int)M.cols, rpc, keys, nf);
    } else {
      const int rpc = 256;
      dim3 grid((unsigned)((M.cols + 255) / 256), (unsigned)((M.rows + rpc - 1) / rpc), (unsigned)count);
      frac_add_keys_cols_kernel<<<grid, 256, 0, S(stream)>>>(static_cast<bf16*>(M.ptr), M.ld, M.stride,
                                                             static_cast<const bf16*>(G.ptr), G.ld, G.stride,
                                                             (int)M.rows, (int)M.cols, rpc, keys, nf);
    }
  }
  return check_launch("frac_add_keys", err);
}

int launch_keys_only(const MatRef& M, int64_t count, int trans, unsigned long long* keys, int* nf, void* stream,
                     std::string* err) {
  const int64_t nkeys = trans ? M.cols : M.rows;
  cudaMemsetAsync(keys, 0, sizeof(unsigned long long) * KEY_DIGITS * nkeys * count, S(stream));
  cudaMemsetAsync(nf, 0, sizeof(int) * nkeys * count, S(stream));
  const int chunk = 256;
  if (!trans) {
    dim3 grid((unsigned)((M.cols + (long long)chunk * 64 - 1) / ((long long)chunk * 64)), (unsigned)M.rows,
              (unsigned)count);
    keys_only_kernel<<<grid, 64, 0, S(stream)>>>(static_cast<const bf16*>(M.ptr), M.ld, M.stride, (int)M.rows,
                                                 (int)M.cols, 0, chunk, keys, nf);
  } else {
    dim3 grid((unsigned)((M.cols + 255) / 256), (unsigned)((M.rows + chunk - 1) / chunk), (unsigned)count);
    keys_only_kernel<<<grid, 256, 0, S(stream)>>>(static_cast<const bf16*>(M.ptr), M.ld, M.stride, (int)M.rows,
                                                  (int)M.cols, 1, chunk, keys, nf);
  }
  return check_launch("keys", err);
}

int launch_select_topk(unsigned long long* keys, const int* nf, int64_t n, int64_t k, int64_t count, int* idx,
                       void* stream, std::string* err) {
  if (n > MAX_SELECT_N) {
    *err = "selection dimension exceeds the supported maximum";
    return GNS_ERR_UNSUPPORTED;
  }
  static bool attr = false;
  if (!attr) {
    cudaFuncSetAttribute(select_topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, MAX_SELECT_N);
    attr = true;
  }
  select_topk_kernel<<<(unsigned)count, 1024, (size_t)n, S(stream)>>>(keys, nf, (int)n, (int)k, idx);
  return check_launch("select_topk", err);
}

int launch_gather(const MatRef& M, int64_t count, int trans, const int* idx, int64_t k, const MatRef& X,
                  float* partials, void* stream, std::string* err, bool decay, float mu, float* bpart) {
  if (!trans) {
    dim3 grid(NPART, (unsigned)count);
    gather_rows_kernel<<<grid, 256, 0, S(stream)>>>(static_cast<bf16*>(M.ptr), M.ld, M.stride, idx, (int)k,
                                                    (int)M.cols, static_cast<bf16*>(X.ptr), X.ld, X.stride, NPART,
                                                    partials, decay ? 1 : 0, mu);
  } else {
    dim3 grid((unsigned)((k + 31) / 32), (unsigned)((M.rows + COL_TILE_ROWS - 1) / COL_TILE_ROWS), (unsigned)count);
    gather_cols_kernel<COL_TILE_ROWS><<<grid, 256, 0, S(stream)>>>(static_cast<bf16*>(M.ptr), M.ld, M.stride, idx, (int)k,
                                                    (int)M.rows, static_cast<bf16*>(X.ptr), X.ld, X.stride,
                                                    decay ? 1 : 0, mu, bpart);
    if (partials && !bpart) {
      MatRef xs = X;
      xs.rows = k;
      xs.cols = M.rows;
      int rc = launch_sumsq(GNS_BF16, xs, count, partials, stream, err);
      if (rc) return rc;
    }
  }
  return check_launch("gather", err);
}

int launch_scale_unselected(const MatRef& W, int64_t count, int trans, const int* idx, int64_t k, float factor,
                            int* flags, void* stream, std::string* err) {
  const int64_t n = trans ? W.cols : W.rows;
  cudaMemsetAsync(flags, 0, sizeof(int) * n * count, S(stream));
  mark_selected_kernel<<<(unsigned)((k * count + 255) / 256), 256, 0, S(stream)>>>(idx, (int)k, (int)n, (int)count,
                                                                                  flags);
  int rc = check_launch("mark_selected", err);
  if (rc) return rc;
  dim3 grid((unsigned)((W.rows + ROWS_PER_BLOCK - 1) / ROWS_PER_BLOCK), (unsigned)count);
  scale_unselected_kernel<<<grid, 256, 0, S(stream)>>>(static_cast<bf16*>(W.ptr), W.ld, W.stride, (int)W.rows,
                                                       (int)W.cols, flags, trans, factor);
  return check_launch("scale_unselected", err);
}

int launch_scatter_update(const MatRef& W, const MatRef& O, int64_t count, int trans, const int* idx, int64_t k,
                          float alpha, float beta, void* stream, std::string* err, const float* rs) {
  const int64_t len = O.cols;
  if (!trans) {
    dim3 grid((unsigned)k, (unsigned)count);
    scatter_update_rows_kernel<<<grid, 256, 0, S(stream)>>>(static_cast<bf16*>(W.ptr), W.ld, W.stride,
                                                            static_cast<const bf16*>(O.ptr), O.ld, O.stride, idx, rs,
                                                            (int)k, (int)len, alpha, beta);
  } else {
    dim3 grid((unsigned)((k + 31) / 32), (unsigned)((len + COL_TILE_ROWS - 1) / COL_TILE_ROWS), (unsigned)count);
    scatter_update_cols_kernel<COL_TILE_ROWS><<<grid, 256, 0, S(stream)>>>(static_cast<bf16*>(W.ptr), W.ld, W.stride,
                                                            static_cast<const bf16*>(O.ptr), O.ld, O.stride, idx, rs,
                                                            (int)k, (int)len, alpha, beta);
  }
  return check_launch("scatter_update", err);
}

int launch_scatter_update_cols_t(const MatRef& W, const MatRef& OT, int64_t count, const int* idx, int64_t k,
                                 float alpha, float beta, void* stream, std::string* err) {
  const int64_t len = OT.rows;
  dim3 grid((unsigned)((k + 31) / 32), (unsigned)((len + COL_TILE_ROWS - 1) / COL_TILE_ROWS), (unsigned)count);
  scatter_update_cols_t_kernel<COL_TILE_ROWS><<<grid, 256, 0, S(stream)>>>(
      static_cast<bf16*>(W.ptr), W.ld, W.stride, static_cast<const bf16*>(OT.ptr), OT.ld, OT.stride, idx, (int)k,
      (int)len, alpha, beta);
  return check_launch("scatter_update_cols_t", err);
}

int launch_row_sumsq(const MatRef& X, int64_t k, int64_t cols, int64_t count, float* s, void* stream,
                     std::string* err) {
  const long long rows = (long long)k * count;
  row_sumsq_kernel<<<(unsigned)((rows + 7) / 8), 256, 0, S(stream)>>>(static_cast<const bf16*>(X.ptr), X.ld, X.stride,
                                                                      (int)k, (int)cols, (int)count, s);
  return check_launch("row_sumsq", err);
}

int launch_col_sumsq(const MatRef& M, int64_t count, float* part, float* s, void* stream, std::string* err) {
  dim3 grid((unsigned)((M.cols + 255) / 256), NPART, (unsigned)count);
  col_sumsq_part_kernel<<<grid, 256, 0, S(stream)>>>(static_cast<const bf16*>(M.ptr), M.ld, M.stride, (int)M.rows,
                                                     (int)M.cols, NPART, part);
  int rc = check_launch("col_sumsq", err);
  if (rc) return rc;
  const long long n = (long long)M.cols * count;
  col_sumsq_finish_kernel<<<(unsigned)((n + 255) / 256), 256, 0, S(stream)>>>(part, (int)M.cols, NPART, (int)count,
                                                                             s);
  return check_launch("col_sumsq_finish", err);
}

int launch_normuon_rows(const float* s, const MatRef& V, const int* idx, int64_t k, int64_t len, int64_t count,
                        float beta2, float eps, float* r, void* stream, std::string* err) {
  normuon_rows_kernel<<<(unsigned)count, 256, 0, S(stream)>>>(s, static_cast<float*>(V.ptr), V.ld, V.stride, idx,
                                                              (int)k, (int)len, beta2, eps, r);
  return check_launch("normuon_rows", err);
}

bool rownorm_fused_supported(int64_t cols) { return cols % 8 == 0 && cols <= 2048 * 8; }

int launch_rownorm_fused_rows(const MatRef& M, const MatRef& G, const MatRef& W, int64_t count, float mu, float gamma,
                              float eps, float alpha, float beta, void* stream, std::string* err) {
  dim3 grid((unsigned)M.rows, (unsigned)count);
  const int vpt = (int)((M.cols + 2047) / 2048);
#define GNS_RN_ARGS                                                                                             \
  static_cast<bf16*>(M.ptr), M.ld, M.stride, static_cast<const bf16*>(G.ptr), G.ld, G.stride,                 \
      static_cast<bf16*>(W.ptr), W.ld, W.stride, (int)M.cols, mu, gamma, eps, alpha, beta
  if (vpt <= 1)
    rownorm_fused_rows_kernel<1><<<grid, 256, 0, S(stream)>>>(GNS_RN_ARGS);
  else if (vpt <= 2)
    rownorm_fused_rows_kernel<2><<<grid, 256, 0, S(stream)>>>(GNS_RN_ARGS);
  else if (vpt <= 4)
    rownorm_fused_rows_kernel<4><<<grid, 256, 0, S(stream)>>>(GNS_RN_ARGS);
  else
    rownorm_fused_rows_kernel<8><<<grid, 256, 0, S(stream)>>>(GNS_RN_ARGS);
#undef GNS_RN_ARGS
  return check_launch("rownorm_fused_rows", err);
}

int launch_rownorm_scale(const float* s, int64_t n, float gamma, float eps, float* r, void* stream,
                         std::string* err) {
  rownorm_scale_kernel<<<(unsigned)((n + 255) / 256), 256, 0, S(stream)>>>(s, (long long)n, gamma, eps, r);
  return check_launch("rownorm_scale", err);
}

int launch_rowscale_update(const MatRef& W, const MatRef& Y, const float* r, int64_t count, int trans, float alpha,
                           float beta, void* stream, std::string* err) {
  dim3 grid((unsigned)((W.rows + ROWS_PER_BLOCK - 1) / ROWS_PER_BLOCK), (unsigned)count);
  rowscale_update_kernel<<<grid, 256, 0, S(stream)>>>(static_cast<bf16*>(W.ptr), W.ld, W.stride,
                                                      static_cast<const bf16*>(Y.ptr), Y.ld, Y.stride, r, (int)W.rows,
                                                      (int)W.cols, trans, alpha, beta);
  return check_launch("rowscale_update", err);
}

int launch_cast_scaled(const MatRef& X16, const MatRef& M, const float* inv, int64_t count, void* stream,
                       std::string* err) {
  dim3 grid((unsigned)((M.rows + ROWS_PER_BLOCK - 1) / ROWS_PER_BLOCK), (unsigned)count);
  cast_scaled_kernel<<<grid, 256, 0, S(stream)>>>(static_cast<__half*>(X16.ptr), X16.ld, X16.stride,
                                                  static_cast<const bf16*>(M.ptr), M.ld, M.stride, inv, (int)M.rows,
                                                  (int)M.cols);
  return check_launch("cast_scaled", err);
}

int launch_axpby(gns_dtype dt, const MatRef& W, const MatRef& Y, int64_t count, float alpha, float beta, void* stream,
                 std::string* err, gns_dtype y_dt) {
  dim3 grid((unsigned)((W.rows + ROWS_PER_BLOCK - 1) / ROWS_PER_BLOCK), (unsigned)count);
  if ((int)y_dt < 0) y_dt = dt;
  if (dt == GNS_BF16 && y_dt == GNS_BF16)
    axpby_kernel<bf16, bf16><<<grid, 256, 0, S(stream)>>>(static_cast<bf16*>(W.ptr), W.ld, W.stride,
                                                         static_cast<const bf16*>(Y.ptr), Y.ld, Y.stride, (int)W.rows,
                                                         (int)W.cols, alpha, beta);
  else if (dt == GNS_BF16 && y_dt == GNS_F16)
    axpby_kernel<bf16, __half><<<grid, 256, 0, S(stream)>>>(static_cast<bf16*>(W.ptr), W.ld, W.stride,
                                                           static_cast<const __half*>(Y.ptr), Y.ld, Y.stride,
                                                           (int)W.rows, (int)W.cols, alpha, beta);
  else if (dt == GNS_F16 && y_dt == GNS_F16)
    axpby_kernel<__half, __half><<<grid, 256, 0, S(stream)>>>(static_cast<__half*>(W.ptr), W.ld, W.stride,
                                                             static_cast<const __half*>(Y.ptr), Y.ld, Y.stride,
                                                             (int)W.rows, (int)W.cols, alpha, beta);
  else if (dt == GNS_F32 && y_dt == GNS_F32)
    axpby_kernel<float, float><<<grid, 256, 0, S(stream)>>>(static_cast<float*>(W.ptr), W.ld, W.stride,
                                                           static_cast<const float*>(Y.ptr), Y.ld, Y.stride,
                                                           (int)W.rows, (int)W.cols, alpha, beta);
  else {
    *err = "internal: unsupported axpby types";
    return GNS_ERR_INVALID;
  }
  return check_launch("axpby", err);
}

int launch_copy(gns_dtype dt, const MatRef& D, const MatRef& Sr, int64_t count, void* stream, std::string* err) {
  dim3 grid(grid_1d(D.rows * D.cols, 256), 1, (unsigned)count);
  if (dt == GNS_BF16 || dt == GNS_F16)  // 16-bit copies move bit patterns
    copy_kernel<uint16_t><<<grid, 256, 0, S(stream)>>>(static_cast<uint16_t*>(D.ptr), D.ld, D.stride,
                                                      static_cast<const uint16_t*>(Sr.ptr), Sr.ld, Sr.stride,
                                                      (int)D.rows, (int)D.cols);
  else
    copy_kernel<float><<<grid, 256, 0, S(stream)>>>(static_cast<float*>(D.ptr), D.ld, D.stride,
                                                   static_cast<const float*>(Sr.ptr), Sr.ld, Sr.stride, (int)D.rows,
                                                   (int)D.cols);
  return check_launch("copy", err);
}

int launch_selftest_wait(const int* counter, int target, uint64_t limit_ns, int* status, unsigned long long* out,
                         void* stream, std::string* err) {
  selftest_wait_kernel<<<1, 32, 0, S(stream)>>>(counter, target, (unsigned long long)limit_ns, status, out);
  return check_launch("selftest_wait", err);
}

}  // namespace gns
