// stream.cu -- the block-FMA stream: one vector set (a[0..k-1], b[0..k-1], c)
// per thread, eq. (1) of "Accurate Models of AMD Matrix Cores" under the model.
//
// The data are read once, so the kernel is a grid-stride stream of 8-, 16- or
// 32-byte vector loads with the evict-first cache hint.  The work per vector is
// integer ALU (decode, significand products, max, shifts, one normalisation) for the
// alignment models; exact-then-round runs on the FP32 pipe (exact products, TwoSum)
// and leaves the sets it does not decide to the integer path, batched per warp.
#include <cuda_runtime.h>

#include <type_traits>

#include "core.cuh"
#include "stream_pair.cuh"

namespace mcemu {

// container sizes: CT 1/2/4 = bytes per element (4 = XF32-style, <= 11-bit
// significands), CT 5 = full binary32 inputs (48-bit significand products)
template <int CT> struct CtBytes { static constexpr int v = CT == 5 ? 4 : CT; };

template <int NB>
__device__ __forceinline__ void load_words(const uint8_t *p, uint32_t (&w)[(NB + 3) / 4]) {
  if constexpr (NB == 1) {
    w[0] = __ldcs(p);
  } else if constexpr (NB == 2) {
    w[0] = __ldcs(reinterpret_cast<const unsigned short *>(p));
  } else if constexpr (NB == 4) {
    w[0] = __ldcs(reinterpret_cast<const unsigned int *>(p));
  } else if constexpr (NB == 8) {
    uint2 v = __ldcs(reinterpret_cast<const uint2 *>(p));
    w[0] = v.x; w[1] = v.y;
  } else {
#pragma unroll
    for (int i = 0; i < NB / 16; i++) {
      uint4 v = __ldcs(reinterpret_cast<const uint4 *>(p) + i);
      w[4 * i] = v.x; w[4 * i + 1] = v.y; w[4 * i + 2] = v.z; w[4 * i + 3] = v.w;
    }
  }
}

template <int ESZ, int K, int NW>
__device__ __forceinline__ void split_elems(const uint32_t (&w)[NW], uint32_t (&e)[K], int nt) {
#pragma unroll
  for (int l = 0; l < K; l++) {
    uint32_t x = 0;
    if (l < nt) {
      if constexpr (ESZ == 1) x = (w[l / 4] >> (8 * (l % 4))) & 0xFFu;
      else if constexpr (ESZ == 2) x = (w[l / 2] >> (16 * (l % 2))) & 0xFFFFu;
      else x = w[l];
    }
    e[l] = x;
  }
}

// Integer formats (INT8/UINT8): exact int32 dot product plus c.
template <int KM>
__global__ void __launch_bounds__(256) block_int_kernel(const __grid_constant__ DevModel m, size_t n,
                                                        const uint8_t *__restrict__ a,
                                                        const uint8_t *__restrict__ b,
                                                        const uint32_t *__restrict__ c,
                                                        uint32_t *__restrict__ d) {
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  const bool ss = m.fa.is_signed && m.fb.is_signed, uu = !m.fa.is_signed && !m.fb.is_signed;
  // software pipeline: the next vector set is loaded while this one is reduced
  uint32_t na[KM / 4], nb[KM / 4], nc = 0;
  size_t v = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (v < n) {
    load_words<KM>(a + v * KM, na);
    load_words<KM>(b + v * KM, nb);
    nc = __ldcs(c + v);
  }
  for (; v < n; v += stride) {
    uint32_t wa[KM / 4], wb[KM / 4];
#pragma unroll
    for (int i = 0; i < KM / 4; i++) { wa[i] = na[i]; wb[i] = nb[i]; }
    const uint32_t cb = nc;
    if (v + stride < n) {
      load_words<KM>(a + (v + stride) * KM, na);
      load_words<KM>(b + (v + stride) * KM, nb);
      nc = __ldcs(c + v + stride);
    }
    int32_t s = 0;       // exact: |sum| <= 32 * 255 * 255
    if (ss) {
#pragma unroll
      for (int i = 0; i < KM / 4; i++) s = __dp4a((int)wa[i], (int)wb[i], s);
    } else if (uu) {
#pragma unroll
      for (int i = 0; i < KM / 4; i++) s = (int32_t)__dp4a(wa[i], wb[i], (unsigned)s);
    } else {
      uint32_t ea[KM], eb[KM];
      split_elems<1, KM>(wa, ea, KM);
      split_elems<1, KM>(wb, eb, KM);
      s = (int32_t)block_int<KM>(m, ea, eb, KM, 0u);
    }
    uint32_t r;
    if (m.int_sat) {
      int64_t t = (int64_t)s + (int64_t)(int32_t)cb;
      t = t > INT32_MAX ? INT32_MAX : (t < INT32_MIN ? INT32_MIN : t);
      r = (uint32_t)(int32_t)t;
    } else {
      r = (uint32_t)s + cb;
    }
    __stcs(d + v, r);
  }
}

// INT8 x INT8 or UINT8 x UINT8 at K = 16, two vector sets per thread and iteration
// (32 bytes of a and of b, 8 of c and d): twice the bytes in flight of block_int_kernel,
// whose one set per thread leaves the stream waiting on memory latency.
__device__ __forceinline__ uint32_t int16_dot(const uint4 &x, const uint4 &y, uint32_t cb, bool ss, bool sat) {
  int32_t s = 0;
  if (ss) {
    s = __dp4a((int)x.x, (int)y.x, s); s = __dp4a((int)x.y, (int)y.y, s);
    s = __dp4a((int)x.z, (int)y.z, s); s = __dp4a((int)x.w, (int)y.w, s);
  } else {
    uint32_t u = 0;
    u = __dp4a(x.x, y.x, u); u = __dp4a(x.y, y.y, u); u = __dp4a(x.z, y.z, u); u = __dp4a(x.w, y.w, u);
    s = (int32_t)u;
  }
  if (sat) {
    int64_t t = (int64_t)s + (int64_t)(int32_t)cb;
    t = t > INT32_MAX ? INT32_MAX : (t < INT32_MIN ? INT32_MIN : t);
    return (uint32_t)(int32_t)t;
  }
  return (uint32_t)s + cb;
}

__global__ void __launch_bounds__(256) int16_pair_kernel(const __grid_constant__ DevModel m, uint32_t npairs,
                                                         const uint4 *__restrict__ a, const uint4 *__restrict__ b,
                                                         const uint2 *__restrict__ c, uint2 *__restrict__ d) {
  const bool ss = m.fa.is_signed != 0, sat = m.int_sat != 0;
  const uint32_t stride = gridDim.x * blockDim.x;
  uint32_t p = blockIdx.x * blockDim.x + threadIdx.x;
  uint4 na0 = {}, na1 = {}, nb0 = {}, nb1 = {};
  uint2 nc = {};
  if (p < npairs) {
    na0 = __ldcs(a + 2 * p); na1 = __ldcs(a + 2 * p + 1);
    nb0 = __ldcs(b + 2 * p); nb1 = __ldcs(b + 2 * p + 1);
    nc = __ldcs(c + p);
  }
  for (; p < npairs; p += stride) {
    const uint4 xa0 = na0, xa1 = na1, xb0 = nb0, xb1 = nb1;
    const uint2 xc = nc;
    const uint32_t q = p + stride;
    if (q < npairs) {
      na0 = __ldcs(a + 2 * q); na1 = __ldcs(a + 2 * q + 1);
      nb0 = __ldcs(b + 2 * q); nb1 = __ldcs(b + 2 * q + 1);
      nc = __ldcs(c + q);
    }
    __stcs(d + p, make_uint2(int16_dot(xa0, xb0, xc.x, ss, sat), int16_dot(xa1, xb1, xc.y, ss, sat)));
  }
}

// Specialised kernel: architecture, format and block size fixed at compile time.
template <int ARCH, int ID, int KM, bool WIDE>
__device__ __forceinline__ uint32_t fast_one(const DevModel &m, const uint8_t *__restrict__ a,
                                             const uint8_t *__restrict__ b, const uint32_t *__restrict__ c,
                                             size_t v) {
  constexpr int NB = KM * Fmt<ID>::BYTES;
  constexpr int NW = (NB + 3) / 4;
  using UT = typename std::conditional<(WIDE || ID == F_FP32), uint64_t, uint32_t>::type;
  using AT = typename std::conditional<(WIDE || ID == F_FP32), int64_t, int32_t>::type;
  uint32_t wa[NW], wb[NW];
  load_words<NB>(a + v * NB, wa);
  load_words<NB>(b + v * NB, wb);
  const uint32_t cb = __ldcs(c + v);
  uint32_t ea[KM], eb[KM];
#pragma unroll
  for (int l = 0; l < KM; l++) {
    ea[l] = felem<ID>(wa, l);
    eb[l] = felem<ID>(wb, l);
  }
  // a queued set has an Inf/NaN operand or addend, so its result is special (the
  // CDNA 3 product overflow can add an infinity: that case takes the whole path)
  constexpr bool kOvf = ID == F_BF16 || ID == F_XF32T || ID == F_XF32R || ID == F_FP32;
  if (!(kOvf && m.prod_ovf)) {
    const uint32_t spec = fspecial_bits<ID, KM>(m, ea, eb, cb);
    if (spec) return resolve_special(m, spec);
  }
  return block_fma_fast<ARCH, ID, KM, UT, AT>(m, ea, eb, cb, true);
}

// One vector set per thread, output rounding RM (1 RNE, 0 toward zero, -1 from the
// model).  A set with an Inf/NaN operand or addend is not evaluated in place: its
// index joins a per-warp queue in shared memory, and each time 32 have gathered the
// warp evaluates them together, so the special-value path runs with every lane busy
// instead of as a divergent branch in nearly every warp.  An exact sum that the
// 64-bit window does not decide joins a second queue of its own, so that the
// full-width evaluator, too, only runs on 32 sets at a time.
constexpr int kStreamThreads = 256;

template <int ARCH, int ID, int KM, bool WIDE, int RM>
__global__ void __launch_bounds__(kStreamThreads) fast_kernel(const __grid_constant__ DevModel m, size_t n,
                                                              const uint8_t *__restrict__ a,
                                                              const uint8_t *__restrict__ b,
                                                              const uint32_t *__restrict__ c,
                                                              uint32_t *__restrict__ d, const W16Consts kc) {
  constexpr int NB = KM * Fmt<ID>::BYTES;
  constexpr int NW = (NB + 3) / 4;
  constexpr bool kWords = Fmt<ID>::BYTES == 2 && Fmt<ID>::XF == 0;   // packed 16-bit decode
  // exact-then-round of FP16 sets on the FP32 pipe first (exact_fp32_sum)
  constexpr bool kFp32Exact = ARCH == MCEMU_ARCH_EXACT && ID == F_FP16;
  // BF16 and truncated XF32 exact-then-round on the FP32 pipe with every term rescaled
  // (exact_scaled)
  constexpr bool kScaled = ARCH == MCEMU_ARCH_EXACT && (ID == F_BF16 || ID == F_XF32T);
  constexpr bool kDefer = ARCH == MCEMU_ARCH_EXACT && (ID == F_FP16 || ID == F_BF16 || ID == F_XF32T ||
                                                       ID == F_XF32R);
  __shared__ size_t queue[kStreamThreads / 32][64];
  __shared__ size_t slow_queue[kDefer ? kStreamThreads / 32 : 1][64];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t below = (1u << lane) - 1u;
  size_t *q = queue[warp], *qs = slow_queue[kDefer ? warp : 0];
  int qn = 0, qsn = 0;                                 // warp-uniform queue lengths
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  // software pipeline: the next vector set's words are loaded while this one is evaluated
  uint32_t na[NW], nb[NW], nc = 0;
  size_t base = (size_t)blockIdx.x * blockDim.x + (size_t)warp * 32;
  if (base + lane < n) {
    load_words<NB>(a + (base + lane) * NB, na);
    load_words<NB>(b + (base + lane) * NB, nb);
    nc = __ldcs(c + base + lane);
  }
  for (; base < n; base += stride) {
    const size_t v = base + lane;
    uint32_t wa[NW], wb[NW];
#pragma unroll
    for (int i = 0; i < NW; i++) { wa[i] = na[i]; wb[i] = nb[i]; }
    const uint32_t cb = nc;
    const size_t vn = v + stride;
    if (vn < n) {
      load_words<NB>(a + vn * NB, na);
      load_words<NB>(b + vn * NB, nb);
      nc = __ldcs(c + vn);
    }
    bool special = false, slow = false;
    if (kFp32Exact && v < n) {
      float p[KM];
#pragma unroll
      for (int i = 0; i < KM / 2; i++) {
        const float2 fa = __half22float2(*reinterpret_cast<const __half2 *>(&wa[i]));
        const float2 fb = __half22float2(*reinterpret_cast<const __half2 *>(&wb[i]));
        p[2 * i] = __fmul_rn(fa.x, fb.x);
        p[2 * i + 1] = __fmul_rn(fa.y, fb.y);
      }
      uint32_t r = 0u;
      slow = exact_fp32_sum<KM>(p, cb, out_rne<RM>(m), m.nan_bits, r) != 0;
      if (!slow) __stcs(d + v, r);
    } else if (v < n) {
      uint32_t sw = (cb & 0x7F800000u) == 0x7F800000u;
#pragma unroll
      for (int i = 0; i < NW; i++) sw |= fspecial_word<ID>(wa[i]) | fspecial_word<ID>(wb[i]);
      special = sw != 0u;
      bool done = special;
      if constexpr (kScaled) {
        // the rescaled products are exact, so a model that turns products of 2^128 or
        // more into Inf (the CDNA 3 rule) keeps the integer path
        if (!done && !m.prod_ovf) {
          uint32_t r = 0u;
          slow = exact_scaled<ID, KM, NW>(wa, wb, cb, out_rne<RM>(m), r) != 0;
          if (!slow) __stcs(d + v, r);
          done = true;
        }
      }
      if (!done) {
        using UT = typename std::conditional<(WIDE || ID == F_FP32), uint64_t, uint32_t>::type;
        using AT = typename std::conditional<(WIDE || ID == F_FP32), int64_t, int32_t>::type;
        uint32_t r;
        if constexpr (kWords) {
          Term<UT> p[KM];
          fterms_w16<ID, KM, UT>(wa, wb, p, kc);
          r = block_fma_terms<ARCH, ID, KM, UT, AT, RM>(m, p, cb, 0u, kDefer ? &slow : nullptr);
        } else {
          uint32_t ea[KM], eb[KM];
#pragma unroll
          for (int l = 0; l < KM; l++) {
            ea[l] = felem<ID>(wa, l);
            eb[l] = felem<ID>(wb, l);
          }
          r = block_fma_fast<ARCH, ID, KM, UT, AT, RM>(m, ea, eb, cb, false, kDefer ? &slow : nullptr);
        }
        if (!slow) __stcs(d + v, r);
      }
    }
    const uint32_t mask = __ballot_sync(0xFFFFFFFFu, special);
    if (mask) {
      if (special) q[qn + __popc(mask & below)] = v;
      qn += __popc(mask);
      if (qn >= 32) {
        __syncwarp();
        const size_t u = q[qn - 32 + lane];
        __stcs(d + u, fast_one<ARCH, ID, KM, WIDE>(m, a, b, c, u));
        qn -= 32;
        __syncwarp();
      }
    }
    if constexpr (kDefer) {
      const uint32_t smask = __ballot_sync(0xFFFFFFFFu, slow);
      if (smask) {
        if (slow) qs[qsn + __popc(smask & below)] = v;
        qsn += __popc(smask);
        if (qsn >= 32) {
          __syncwarp();
          const size_t u = qs[qsn - 32 + lane];
          __stcs(d + u, fast_one<ARCH, ID, KM, WIDE>(m, a, b, c, u));
          qsn -= 32;
          __syncwarp();
        }
      }
    }
  }
  __syncwarp();
  if (lane < qn) {
    const size_t u = q[lane];
    __stcs(d + u, fast_one<ARCH, ID, KM, WIDE>(m, a, b, c, u));
  }
  if (kDefer && lane < qsn) {
    const size_t u = qs[lane];
    __stcs(d + u, fast_one<ARCH, ID, KM, WIDE>(m, a, b, c, u));
  }
}

// The pair kernel serves, on 8-byte sets (FP16/BF16 K=4, truncated XF32 K=2) with kept
// subnormals:
//  - early-c global alignment with truncated alignment, F_p >= 23 (P0, P0c >= 0),
//    32-bit sums, no exponent limit and c = 0 discarded;
//  - exact-then-round without the CDNA 3 product-overflow rule;
// with operand pointers 16-byte aligned and c, d 8-byte aligned.
static bool pair_ok(const DevModel &m, int id, const void *a, const void *b, const uint32_t *c, const uint32_t *d) {
  if (!((id == F_FP16 || id == F_BF16) && m.k == 4) && !(id == F_XF32T && m.k == 2)) return false;
  if (m.acc16 || m.sub_out_flush || m.fa.sub_keep == 0u || m.c_sub_keep == 0u || m.prod_ovf) return false;
  if (m.arch == MCEMU_ARCH_GA_EARLY) {
    if (m.align_rd || m.wide || m.emin_lim != kNegE || m.c_zero_exp != kNegE || m.R0 != 0 || m.R0c != 0) return false;
  } else if (m.arch != MCEMU_ARCH_EXACT) {
    return false;
  }
  return ((uintptr_t)a % 16) == 0 && ((uintptr_t)b % 16) == 0 && ((uintptr_t)c % 8) == 0 && ((uintptr_t)d % 8) == 0;
}

static int grid_for(size_t n, const void *kernel);

static int launch_pair(const DevModel &m, int id, size_t n, const void *a, const void *b, const uint32_t *c,
                       uint32_t *d, cudaStream_t s) {
  const int mb = id == F_BF16 ? 7 : 10;            // kE: the 16-bit formats' exponent extraction
  const GaPairK k{m.p0mul, m.p0cmul, -2 * m.fa.bias - m.F, 1u, 2u, 1u << 16, 1u << (16 - mb), 1u << 9, 1u << 23, -1, -2,
                  1u << 24, 1u << 22};
  const size_t np = n / 2;
  auto run = [&](auto kern) {
    const int grid = grid_for(np, (const void *)kern);
    kern<<<grid, kPairThreads, 0, s>>>(m, (uint32_t)np, (const uint4 *)a, (const uint4 *)b, (const uint2 *)c,
                                       (uint2 *)d, k);
    return cudaGetLastError() == cudaSuccess ? MCEMU_OK : MCEMU_ERR_CUDA;
  };
  auto by_rm = [&](auto id_tag, auto exact_tag) {
    constexpr int ID = decltype(id_tag)::value;
    if constexpr (decltype(exact_tag)::value)
      return m.rne ? run(pair_kernel<ExactPairEv<ID, 1>>) : run(pair_kernel<ExactPairEv<ID, 0>>);
    else
      return m.rne ? run(pair_kernel<GaPairEv<ID, 1>>) : run(pair_kernel<GaPairEv<ID, 0>>);
  };
  using T = std::true_type;
  using Fl = std::false_type;
  const bool ex = m.arch == MCEMU_ARCH_EXACT;
  if (id == F_BF16) return ex ? by_rm(std::integral_constant<int, F_BF16>{}, T{}) : by_rm(std::integral_constant<int, F_BF16>{}, Fl{});
  if (id == F_XF32T) return ex ? by_rm(std::integral_constant<int, F_XF32T>{}, T{}) : by_rm(std::integral_constant<int, F_XF32T>{}, Fl{});
  return ex ? by_rm(std::integral_constant<int, F_FP16>{}, T{}) : by_rm(std::integral_constant<int, F_FP16>{}, Fl{});
}

// Any model: element loads, the out-of-line evaluator (the fallback for
// combinations without a specialised kernel).
__global__ void __launch_bounds__(256) block_generic_kernel(const __grid_constant__ DevModel m, size_t n, int eb,
                                                            const uint8_t *__restrict__ a,
                                                            const uint8_t *__restrict__ b,
                                                            const uint32_t *__restrict__ c,
                                                            uint32_t *__restrict__ d) {
  const int k = m.k;
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  for (size_t v = (size_t)blockIdx.x * blockDim.x + threadIdx.x; v < n; v += stride) {
    uint32_t ea[32], ebv[32];
    for (int l = 0; l < k; l++) {
      size_t idx = v * k + l;
      if (eb == 1) { ea[l] = a[idx]; ebv[l] = b[idx]; }
      else if (eb == 2) { ea[l] = reinterpret_cast<const uint16_t *>(a)[idx]; ebv[l] = reinterpret_cast<const uint16_t *>(b)[idx]; }
      else { ea[l] = reinterpret_cast<const uint32_t *>(a)[idx]; ebv[l] = reinterpret_cast<const uint32_t *>(b)[idx]; }
    }
    d[v] = block_eval_generic(m, ea, ebv, k, c[v]);
  }
}

// ---------------------------------------------------------------------------
// dispatch: specialised kernels for the block sizes and formats of the
// workloads and the hardware presets; everything else takes the generic kernel
// ---------------------------------------------------------------------------
static int grid_for(size_t n, const void *kernel) {
  // resident blocks per SM and the SM count, looked up once per (device, kernel) and
  // thread: a short launch is otherwise dominated by the queries
  struct Entry {
    const void *kernel;
    int dev, sms, per_sm;
  };
  static thread_local Entry cache[64];
  static thread_local int cached = 0;
  int dev = 0, sms = 0, per_sm = 0;
  cudaGetDevice(&dev);
  for (int i = 0; i < cached; i++)
    if (cache[i].kernel == kernel && cache[i].dev == dev) {
      sms = cache[i].sms;
      per_sm = cache[i].per_sm;
      break;
    }
  if (sms == 0) {
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, 256, 0);
    if (cached < 64) cache[cached++] = Entry{kernel, dev, sms, per_sm};
  }
  if (per_sm < 1) per_sm = 1;
  size_t want = (n + 255) / 256;
  size_t full = (size_t)sms * per_sm;              // one wave of resident blocks
  if (want > full) want = full;
  return (int)(want < 1 ? 1 : want);
}

typedef void (*FpKernel)(const DevModel, size_t, const uint8_t *, const uint8_t *, const uint32_t *, uint32_t *,
                         const W16Consts);

struct Special {
  int arch, id, km, wide, rm;                          // rm: output rounding, -1 = any
  FpKernel fn;
};

#define SPEC(A, F, K, W) {A, F, K, W, -1, fast_kernel<A, F, K, W, -1>}
#define SPEC_RM(A, F, K) {A, F, K, false, 0, fast_kernel<A, F, K, false, 0>}, \
                         {A, F, K, false, 1, fast_kernel<A, F, K, false, 1>}
static const Special kSpecial[] = {
    // early-c global alignment: the randomized-workload truncate / RNE models
    SPEC_RM(MCEMU_ARCH_GA_EARLY, F_FP16, 4), SPEC_RM(MCEMU_ARCH_GA_EARLY, F_BF16, 4),
    SPEC_RM(MCEMU_ARCH_GA_EARLY, F_XF32T, 2), SPEC(MCEMU_ARCH_GA_EARLY, F_E4M3, 8, false),
    SPEC(MCEMU_ARCH_GA_EARLY, F_E5M2, 8, false),
    // exact-then-round on the same vector sets
    SPEC_RM(MCEMU_ARCH_EXACT, F_FP16, 4), SPEC_RM(MCEMU_ARCH_EXACT, F_BF16, 4),
    SPEC_RM(MCEMU_ARCH_EXACT, F_XF32T, 2), SPEC(MCEMU_ARCH_EXACT, F_E4M3, 8, false),
    SPEC(MCEMU_ARCH_EXACT, F_E5M2, 8, false),
    // CDNA 3: Algorithm 1 (fp16/bf16 N_FMA 8, tf19 4), Algorithm 2 (binary8 FNUZ, 16)
    SPEC(MCEMU_ARCH_GA_LATE, F_FP16, 8, false), SPEC(MCEMU_ARCH_GA_LATE, F_BF16, 8, false),
    SPEC(MCEMU_ARCH_GA_LATE, F_XF32T, 4, false), SPEC(MCEMU_ARCH_ODD_EVEN, F_E4M3Z, 16, false),
    SPEC(MCEMU_ARCH_ODD_EVEN, F_E5M2Z, 16, false),
    // Table 3 NVIDIA-like presets
    SPEC(MCEMU_ARCH_GA_EARLY, F_FP16, 16, true), SPEC(MCEMU_ARCH_GA_EARLY, F_FP16, 8, false),
    SPEC(MCEMU_ARCH_GA_EARLY, F_BF16, 8, false), SPEC(MCEMU_ARCH_GA_EARLY, F_XF32T, 4, false),
};
#undef SPEC
#undef SPEC_RM

// compile-time format of a model whose operands share one format, else -1
static int fmt_id(const DevModel &m) {
  const FmtDev &a = m.fa, &b = m.fb;
  if (a.is_int || a.mbits != b.mbits || a.bias != b.bias || a.xf32 != b.xf32 || a.sw_fnuz != b.sw_fnuz ||
      a.emask != b.emask)
    return -1;
  if (a.xf32) return a.xf32 == 2 ? F_XF32R : F_XF32T;
  if (a.mbits == 23) return F_FP32;
  if (a.mbits == 10) return F_FP16;
  if (a.mbits == 7) return F_BF16;
  if (a.mbits == 3) return a.sw_fnuz ? F_E4M3Z : F_E4M3;
  if (a.mbits == 2) return a.sw_fnuz ? F_E5M2Z : F_E5M2;
  return -1;
}

int launch_block_fma(const DevModel &m, size_t n, const void *a, const void *b, const uint32_t *c,
                     uint32_t *d, void *stream) {
  if (n == 0) return MCEMU_OK;
  cudaStream_t s = (cudaStream_t)stream;
  if (m.fa.is_int && m.k == 16 && m.fa.is_signed == m.fb.is_signed && n >= 2 && n / 2 < (1u << 31) &&
      ((uintptr_t)a % 16) == 0 && ((uintptr_t)b % 16) == 0 && ((uintptr_t)c % 8) == 0 && ((uintptr_t)d % 8) == 0) {
    const int grid = grid_for(n / 2, (const void *)int16_pair_kernel);
    int16_pair_kernel<<<grid, 256, 0, s>>>(m, (uint32_t)(n / 2), (const uint4 *)a, (const uint4 *)b, (const uint2 *)c,
                                           (uint2 *)d);
    if (cudaGetLastError() != cudaSuccess) return MCEMU_ERR_CUDA;
    if (n % 2 == 0) return MCEMU_OK;
    const size_t t = n - 1;                            // the odd last set: the one-set kernel
    return launch_block_fma(m, 1, (const uint8_t *)a + 16 * t, (const uint8_t *)b + 16 * t, c + t, d + t, stream);
  }
  if (m.fa.is_int && (m.k == 16 || m.k == 8 || m.k == 32 || m.k == 4)) {
    auto run = [&](auto kern) {
      int grid = grid_for(n, (const void *)kern);
      kern<<<grid, 256, 0, s>>>(m, n, (const uint8_t *)a, (const uint8_t *)b, c, d);
      return cudaGetLastError() == cudaSuccess ? MCEMU_OK : MCEMU_ERR_CUDA;
    };
    if (m.k == 4) return run(block_int_kernel<4>);
    if (m.k == 8) return run(block_int_kernel<8>);
    if (m.k == 16) return run(block_int_kernel<16>);
    return run(block_int_kernel<32>);
  }
  const int id = fmt_id(m);
  if (id >= 0 && f8_stream_ok(m, id)) return launch_block_fma_f8(m, id, n, a, b, c, d, stream);
  if (id >= 0 && n >= 2 && n / 2 < (1u << 31) && pair_ok(m, id, a, b, c, d)) {
    int st = launch_pair(m, id, n, a, b, c, d, s);
    if (st != MCEMU_OK || n % 2 == 0) return st;
    const size_t t = n - 1, vb = 8;                    // the odd last set: the one-set kernel
    return launch_block_fma(m, 1, (const uint8_t *)a + t * vb, (const uint8_t *)b + t * vb, c + t, d + t, stream);
  }
  // the specialised kernels assume kept subnormals (the fp32 special-value shortcut)
  if (id >= 0 && !m.acc16 && m.arch != MCEMU_ARCH_PAIRWISE && m.fa.sub_keep != 0u && m.c_sub_keep != 0u) {
    for (const Special &sp : kSpecial) {
      if (sp.arch != m.arch || sp.id != id || sp.km != m.k) continue;
      if (m.arch != MCEMU_ARCH_EXACT && sp.wide != (m.wide != 0)) continue;
      if (sp.rm >= 0 && sp.rm != (m.rne != 0 ? 1 : 0)) continue;
      int grid = grid_for(n, (const void *)sp.fn);
      const uint32_t mb = id == F_FP16 ? 10u : 7u;                  // fterms_w16 (FP16, BF16)
      const W16Consts kc{1u, 2u, 1u << 16, 1u << (32 - mb), (1u << 22) - 1u, 1u << 10};
      sp.fn<<<grid, 256, 0, s>>>(m, n, (const uint8_t *)a, (const uint8_t *)b, c, d, kc);
      return cudaGetLastError() == cudaSuccess ? MCEMU_OK : MCEMU_ERR_CUDA;
    }
  }
  const int eb = m.fa.is_int ? 1 : (int)(m.fa.sshift + 1) / 8;
  int grid = grid_for(n, (const void *)block_generic_kernel);
  block_generic_kernel<<<grid, 256, 0, s>>>(m, n, eb, (const uint8_t *)a, (const uint8_t *)b, c, d);
  return cudaGetLastError() == cudaSuccess ? MCEMU_OK : MCEMU_ERR_CUDA;
}

}  // namespace mcemu
