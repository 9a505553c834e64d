// multiword.cu -- multi-word GEMM ("Accurate Models of AMD Matrix Cores",
// Sec. 8.1): binary64 matrices split into BF16 words, every word pair
// multiplied on the emulated matrix unit, the fp32 word products summed in
// binary64.  The word-pair chains of one output run in one thread, and the
// binary64 combine happens in registers in a fixed order (i+j descending, then
// i ascending), so no word-product matrix is ever stored.
#include <cuda_runtime.h>

#include <atomic>
#include <mutex>

#include "core.cuh"

namespace mcemu {

// RNE of a binary64 value to bfloat16 bits (8-bit significand, exponent range of
// binary32, subnormals on the 2^-133 grid, overflow to Inf).
__device__ __forceinline__ uint16_t rne_bf16(double x) {
  uint64_t u = (uint64_t)__double_as_longlong(x);
  uint32_t sign = (uint32_t)(u >> 63) << 15;
  uint32_t ef = (uint32_t)(u >> 52) & 0x7FFu;
  uint64_t mf = u & 0xFFFFFFFFFFFFFull;
  if (ef == 0x7FFu) return (uint16_t)(sign | (mf ? 0x7FC0u : 0x7F80u));
  if (ef == 0 && mf == 0) return (uint16_t)sign;
  // value = M * 2^(E - 52), M with hidden bit (binary64 subnormals keep E = -1022)
  uint64_t M = ef ? (mf | (1ull << 52)) : mf;
  int32_t E = ef ? (int32_t)ef - 1023 : -1022;
  int32_t p = 63 - __clzll((long long)M);            // msb of M
  int32_t Ev = E - 52 + p;                           // exponent of the value
  int32_t Ec = Ev < -126 ? -126 : Ev;
  int32_t r = Ec - 7 - (E - 52);                     // bits of M below the bf16 grid
  uint64_t q;
  uint32_t up = 0;
  if (r <= 0) {
    q = M << (-r);
  } else if (r > 63) {
    q = 0;
  } else {
    q = M >> r;
    uint64_t rem = M & ((1ull << r) - 1ull);
    uint64_t half = 1ull << (r - 1);
    up = (rem > half || (rem == half && (q & 1ull))) ? 1u : 0u;
  }
  if (Ec > 127) return (uint16_t)(sign | 0x7F80u);
  uint32_t bits = ((uint32_t)(Ec + 126) << 7) + (uint32_t)q + up;
  if (bits >= 0x7F80u) bits = 0x7F80u;
  return (uint16_t)(sign | bits);
}

__device__ __forceinline__ double bf16_to_double(uint16_t w) {
  return (double)__uint_as_float((uint32_t)w << 16);
}

// x [rows][ldx] -> words [n_words][rows * cols] (plane stride word_stride)
__global__ void split_kernel(int n_words, int rows, int cols, const double *__restrict__ x, int64_t ldx,
                             uint16_t *__restrict__ words, int64_t word_stride) {
  const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= (int64_t)rows * cols) return;
  const int64_t r = t / cols, q = t % cols;
  double v = x[r * ldx + q];
  for (int w = 0; w < n_words; w++) {
    uint16_t b = rne_bf16(v);
    words[(int64_t)w * word_stride + t] = b;
    v = __dsub_rn(v, bf16_to_double(b));             // exact residual
  }
}

int launch_multiword_split(int n_words, size_t n, const double *x, int64_t ldx, int rows, uint16_t *words,
                           int64_t word_stride, void *stream) {
  cudaStream_t s = (cudaStream_t)stream;
  const int cols = (int)(n / (size_t)rows);
  const int64_t total = (int64_t)rows * cols;
  split_kernel<<<(int)((total + 255) / 256), 256, 0, s>>>(n_words, rows, cols, x, ldx, words, word_stride);
  return cudaGetLastError() == cudaSuccess ? MCEMU_OK : MCEMU_ERR_CUDA;
}

// Fused word-pair GEMM: one output per thread, NW^2 fp32 chains, binary64 combine.
constexpr int kMwTile = 16;

__host__ __device__ __forceinline__ int mw_chunk(int kt) { return kt >= 64 ? kt : kt * (64 / kt); }

template <int NW>
__global__ void __launch_bounds__(kMwTile *kMwTile) multiword_kernel(
    const DevModel m, int kt, int truncated, int M, int N, int K, const uint16_t *__restrict__ Aw,
    const uint16_t *__restrict__ Bw, double *D, int64_t ldd) {
  extern __shared__ uint32_t smem[];
  const int KC = mw_chunk(kt);
  uint32_t *As = smem;                                   // [NW][kMwTile][KC]
  uint32_t *Bs = smem + NW * kMwTile * KC;               // [NW][kMwTile][KC]
  const int i0 = blockIdx.y * kMwTile, j0 = blockIdx.x * kMwTile;
  const int tid = threadIdx.y * kMwTile + threadIdx.x;
  const int ti = threadIdx.y, tj = threadIdx.x;
  uint32_t acc[NW * NW];
  for (int p = 0; p < NW * NW; p++) acc[p] = 0u;        // C = 0
  for (int k0 = 0; k0 < K; k0 += KC) {
    const int kc = min(KC, K - k0);
    __syncthreads();
    for (int e = tid; e < NW * kMwTile * KC; e += kMwTile * kMwTile) {
      int w = e / (kMwTile * KC), r = (e / KC) % kMwTile, q = e % KC;
      int i = i0 + r, j = j0 + r;
      As[e] = (i < M && q < kc) ? Aw[(int64_t)w * M * K + (int64_t)i * K + k0 + q] : 0u;
      Bs[e] = (j < N && q < kc) ? Bw[(int64_t)w * N * K + (int64_t)j * K + k0 + q] : 0u;
    }
    __syncthreads();
    for (int s0 = 0; s0 < kc; s0 += kt) {
      const int send = min(s0 + kt, kc);
      for (int b0 = s0; b0 < send; b0 += m.k) {
        const int nt = min(m.k, send - b0);
        for (int wi = 0; wi < NW; wi++)
          for (int wj = 0; wj < NW; wj++) {
            if (truncated && wi + wj + 2 > NW + 1) continue;
            acc[wi * NW + wj] = block_eval_generic(m, As + (wi * kMwTile + ti) * KC + b0,
                                                   Bs + (wj * kMwTile + tj) * KC + b0, nt, acc[wi * NW + wj]);
          }
      }
    }
  }
  const int i = i0 + ti, j = j0 + tj;
  if (i >= M || j >= N) return;
  double d = 0.0;
  for (int s = 2 * NW; s >= 2; s--)                    // i + j descending (1-based words)
    for (int wi = 1; wi <= NW; wi++) {                 // then i ascending
      const int wj = s - wi;
      if (wj < 1 || wj > NW) continue;
      if (truncated && wi + wj > NW + 1) continue;
      d = __dadd_rn(d, (double)__uint_as_float(acc[(wi - 1) * NW + (wj - 1)]));
    }
  D[(int64_t)i * ldd + j] = d;
}

// D = fl64(D + P) (or fl64(0 + P) for the first word product), P the fp32 bits of one
// word product
__global__ void __launch_bounds__(256) combine_kernel(int M, int N, const uint32_t *__restrict__ P, double *D,
                                                      int64_t ldd, int first) {
  const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= (int64_t)M * N) return;
  double *p = D + (t / N) * ldd + t % N;
  *p = __dadd_rn(first ? 0.0 : *p, (double)__uint_as_float(P[t]));
}

template <int NW>
static int run_mw(const DevModel &m, int kt, int truncated, int M, int N, int K, const uint16_t *Aw,
                  const uint16_t *Bw, double *D, int64_t ldd, cudaStream_t s) {
  const int KC = mw_chunk(kt);
  size_t shm = (size_t)2 * NW * kMwTile * KC * 4;
  auto kern = multiword_kernel<NW>;
  if (shm > 48 * 1024 &&
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)shm) != cudaSuccess)
    return MCEMU_ERR_UNSUPPORTED;
  dim3 grid((N + kMwTile - 1) / kMwTile, (M + kMwTile - 1) / kMwTile), block(kMwTile, kMwTile);
  kern<<<grid, block, shm, s>>>(m, kt, truncated, M, N, K, Aw, Bw, D, ldd);
  return cudaGetLastError() == cudaSuccess ? MCEMU_OK : MCEMU_ERR_CUDA;
}

int launch_multiword_gemm(const DevModel &m, int kt, int n_words, int truncated, int M, int N, int K,
                          const double *A, int64_t lda, const double *Bt, int64_t ldb, double *D, int64_t ldd,
                          void *ws, size_t ws_bytes, void *stream) {
  cudaStream_t s = (cudaStream_t)stream;
  if (n_words > 4 || kt > 256) return MCEMU_ERR_UNSUPPORTED;
  (void)ws_bytes;
  uint16_t *Aw = (uint16_t *)ws;
  size_t wa = ((size_t)n_words * M * K * 2 + 255) & ~(size_t)255;
  uint16_t *Bw = (uint16_t *)((uint8_t *)ws + wa);
  if (K > 0) {
    int st = launch_multiword_split(n_words, (size_t)M * K, A, lda, M, Aw, (int64_t)M * K, stream);
    if (st != MCEMU_OK) return st;
    st = launch_multiword_split(n_words, (size_t)N * K, Bt, ldb, N, Bw, (int64_t)N * K, stream);
    if (st != MCEMU_OK) return st;
  }
  if (gemm_fast_ok(m) && kt <= 64) {
    // one fast tile GEMM per word pair into the fp32 buffer after the words, each
    // added into the binary64 D in the combine order: i + j descending, then i ascending
    const size_t wb = ((size_t)n_words * N * K * 2 + 255) & ~(size_t)255;
    uint32_t *P = (uint32_t *)((uint8_t *)ws + wa + wb);
    int first = 1;
    for (int sum = 2 * n_words; sum >= 2; sum--)
      for (int wi = 1; wi <= n_words; wi++) {
        const int wj = sum - wi;
        if (wj < 1 || wj > n_words || (truncated && wi + wj > n_words + 1)) continue;
        int st = launch_tile_gemm_fast(m, kt, M, N, K, Aw + (size_t)(wi - 1) * M * K, K,
                                       Bw + (size_t)(wj - 1) * N * K, K, nullptr, 0, P, N, stream);
        if (st != MCEMU_OK) return st;
        const int64_t total = (int64_t)M * N;
        combine_kernel<<<(unsigned)((total + 255) / 256), 256, 0, s>>>(M, N, P, D, ldd, first);
        if (cudaGetLastError() != cudaSuccess) return MCEMU_ERR_CUDA;
        first = 0;
      }
    return MCEMU_OK;
  }
  switch (n_words) {
    case 1: return run_mw<1>(m, kt, truncated, M, N, K, Aw, Bw, D, ldd, s);
    case 2: return run_mw<2>(m, kt, truncated, M, N, K, Aw, Bw, D, ldd, s);
    case 3: return run_mw<3>(m, kt, truncated, M, N, K, Aw, Bw, D, ldd, s);
    default: return run_mw<4>(m, kt, truncated, M, N, K, Aw, Bw, D, ldd, s);
  }
}

// ---------------------------------------------------------------------------
// The same GEMM for callers that cannot allocate device memory where they call
// it (a host program that only holds buffers handed to it, a loop whose device
// memory is budgeted up front): the words of A and B go to a fixed array of this
// module's device memory instead of caller workspace.  The split kernel writes
// every word the GEMM kernel reads, and each word product is written before the
// combine reads it, so nothing in the array has to start at zero.  One array per device serves every call: calls whose kernels may
// overlap race on it.
// ---------------------------------------------------------------------------
static __device__ __align__(256) uint8_t g_mw_static_ws[MCEMU_MULTIWORD_STATIC_BYTES];

constexpr int kMaxDevices = 64;
static std::atomic<void *> g_mw_static_ptr[kMaxDevices];
static std::mutex g_mw_static_mu;

// device address of the array on the current device; looked up once per device,
// with that device current (the caller's), then cached
static void *mw_static_ptr(int &status) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) { status = MCEMU_ERR_CUDA; return nullptr; }
  if (dev < 0 || dev >= kMaxDevices) { status = MCEMU_ERR_UNSUPPORTED; return nullptr; }
  void *p = g_mw_static_ptr[dev].load(std::memory_order_acquire);
  if (p) return p;
  std::lock_guard<std::mutex> lock(g_mw_static_mu);
  p = g_mw_static_ptr[dev].load(std::memory_order_relaxed);
  if (!p) {
    if (cudaGetSymbolAddress(&p, g_mw_static_ws) != cudaSuccess || !p) {
      status = MCEMU_ERR_CUDA;
      return nullptr;
    }
    g_mw_static_ptr[dev].store(p, std::memory_order_release);
  }
  return p;
}

int launch_multiword_gemm_static(const DevModel &m, int kt, int n_words, int truncated, int M, int N, int K,
                                 const double *A, int64_t lda, const double *Bt, int64_t ldb, double *D,
                                 int64_t ldd, void *stream) {
  int status = MCEMU_OK;
  void *ws = mw_static_ptr(status);
  if (!ws) return status;
  return launch_multiword_gemm(m, kt, n_words, truncated, M, N, K, A, lda, Bt, ldb, D, ldd, ws,
                               MCEMU_MULTIWORD_STATIC_BYTES, stream);
}

// ||D - R||_F^2 and ||R||_F^2 with a fixed reduction order (deterministic)
constexpr int kFroBlocks = 512;

__global__ void fro_partial(int M, int N, const double *__restrict__ D, int64_t ldd, const double *__restrict__ R,
                            int64_t ldr, double *part) {
  __shared__ double s0[256], s1[256];
  double a = 0.0, b = 0.0;
  const int64_t total = (int64_t)M * N;
  for (int64_t t = (int64_t)blockIdx.x * 256 + threadIdx.x; t < total; t += (int64_t)kFroBlocks * 256) {
    int64_t i = t / N, j = t % N;
    double r = R[i * ldr + j];
    double e = __dsub_rn(D[i * ldd + j], r);
    a = __fma_rn(e, e, a);
    b = __fma_rn(r, r, b);
  }
  s0[threadIdx.x] = a;
  s1[threadIdx.x] = b;
  __syncthreads();
  for (int w = 128; w > 0; w >>= 1) {
    if (threadIdx.x < w) {
      s0[threadIdx.x] += s0[threadIdx.x + w];
      s1[threadIdx.x] += s1[threadIdx.x + w];
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    part[blockIdx.x] = s0[0];
    part[kFroBlocks + blockIdx.x] = s1[0];
  }
}

__global__ void fro_final(const double *part, double *out) {
  __shared__ double s0[256], s1[256];
  double a = 0.0, b = 0.0;
  for (int t = threadIdx.x; t < kFroBlocks; t += 256) {
    a += part[t];
    b += part[kFroBlocks + t];
  }
  s0[threadIdx.x] = a;
  s1[threadIdx.x] = b;
  __syncthreads();
  for (int w = 128; w > 0; w >>= 1) {
    if (threadIdx.x < w) {
      s0[threadIdx.x] += s0[threadIdx.x + w];
      s1[threadIdx.x] += s1[threadIdx.x + w];
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    out[0] = s0[0];
    out[1] = s1[0];
  }
}

int launch_fro_error(int M, int N, const double *D, int64_t ldd, const double *R, int64_t ldr, double *out,
                     void *stream) {
  cudaStream_t s = (cudaStream_t)stream;
  double *part = out + 2;                              // caller scratch: 2 * kFroBlocks doubles
  fro_partial<<<kFroBlocks, 256, 0, s>>>(M, N, D, ldd, R, ldr, part);
  fro_final<<<1, 256, 0, s>>>(part, out);
  return cudaGetLastError() == cudaSuccess ? MCEMU_OK : MCEMU_ERR_CUDA;
}

}  // namespace mcemu
