// api.cu -- the C ABI of libmcemu.so (include/mcemu.h): argument checks, model
// presets and validation, the MFMA/SWMMAC tile helpers, and dispatch into the
// kernels.  No function here computes a result on the host.
#include <cuda_runtime.h>

#include <climits>
#include <cstring>
#include <new>

#include "model.h"

using namespace mcemu;

struct mcemu_model {
  Model m;
};

extern "C" {

const char *mcemu_status_string(int status) {
  switch (status) {
    case MCEMU_OK: return "ok";
    case MCEMU_ERR_INVALID_ARG: return "invalid argument";
    case MCEMU_ERR_UNSUPPORTED: return "unsupported";
    case MCEMU_ERR_NOT_2_4: return "not 2:4 sparse";
    case MCEMU_ERR_ALIGNMENT: return "misaligned pointer or leading dimension";
    case MCEMU_ERR_CUDA: return "CUDA error";
    case MCEMU_ERR_TIMEOUT: return "device wait timed out";
    case MCEMU_ERR_WORKSPACE: return "workspace too small";
    default: return "unknown status";
  }
}

int mcemu_version(void) { return 10000; }

}  // extern "C"

// ---------------------------------------------------------------------------
// presets: the feature vectors of "Accurate Models of AMD Matrix Cores",
// Secs. 4.1-4.3 and Table 3
// ---------------------------------------------------------------------------
static void base_desc(mcemu_model_desc *d, int fmt, int arch, int k) {
  std::memset(d, 0, sizeof *d);
  d->struct_size = sizeof(mcemu_model_desc);
  d->fmt_a = d->fmt_b = fmt;
  d->fp8_enc = MCEMU_FP8_OCP;
  d->xf32_round = MCEMU_XF32_TRUNC;
  d->arch = arch;
  d->block_k = k;
  d->align_frac_bits = 24;
  d->align_round = MCEMU_ALIGN_RZ;
  d->c_frac_bits = 24;
  d->psum_frac_bits = 32;
  d->post_norm_frac_bits = 31;
  d->acc_sig_bits = 24;
  d->out_round = MCEMU_OUT_RNE;
  d->c_zero_exp = MCEMU_NO_EXP;
  d->emin_lim = MCEMU_NO_EXP;
  d->nan_bits = 0x7FC00000u;
  d->pair_group = k;
}

static void cdna3(mcemu_model_desc *d, int fmt, int arch, int k) {
  base_desc(d, fmt, arch, k);
  d->c_zero_exp = -126;        // "c = 0 is considered as subnormal number" (Sec. 4.3.2)
  d->prod_overflow_2p128 = 1;  // |p| >= 2^128 -> Inf (Sec. 4.3.2)
  d->nan_bits = 0xFFC00000u;   // the NaN carries a negative sign
}

static void early(mcemu_model_desc *d, int fmt, int k, int frac, int out, int emin) {
  base_desc(d, fmt, MCEMU_ARCH_GA_EARLY, k);
  d->align_frac_bits = frac;
  d->out_round = out;
  d->emin_lim = emin;
}

// fp16 output (Table 3's note): binary16 c and d, RTZ, the fp16 e_min limit
static void early16(mcemu_model_desc *d, int fmt, int k, int frac, int emin) {
  early(d, fmt, k, frac, MCEMU_OUT_RTZ, emin);
  d->acc_sig_bits = 11;
  d->nan_bits = 0x7E00u;       // the quiet NaN of binary16
}

static void pairwise(mcemu_model_desc *d, int fmt, int group) {
  base_desc(d, fmt, MCEMU_ARCH_PAIRWISE, group);
  d->subnormal_in_flush = 1;
  d->subnormal_out_flush = 1;
  d->nan_bits = 0xFFC00000u;
}

extern "C" int mcemu_model_preset(int preset, int fmt, int block_k, mcemu_model_desc *out) {
  if (!out) return MCEMU_ERR_INVALID_ARG;
  const bool hw = preset < 100;
  if (hw && (fmt != -1 || block_k != 0)) return MCEMU_ERR_INVALID_ARG;
  switch (preset) {
    case MCEMU_PRESET_CDNA3_FP16: cdna3(out, MCEMU_FP16, MCEMU_ARCH_GA_LATE, 8); break;
    case MCEMU_PRESET_CDNA3_BF16: cdna3(out, MCEMU_BF16, MCEMU_ARCH_GA_LATE, 8); break;
    case MCEMU_PRESET_CDNA3_XF32: cdna3(out, MCEMU_XF32, MCEMU_ARCH_GA_LATE, 4); break;
    case MCEMU_PRESET_CDNA3_FP8:
      cdna3(out, MCEMU_E4M3, MCEMU_ARCH_ODD_EVEN, 16);
      out->fp8_enc = MCEMU_FP8_FNUZ;
      break;
    case MCEMU_PRESET_CDNA3_BF8:
      cdna3(out, MCEMU_E5M2, MCEMU_ARCH_ODD_EVEN, 16);
      out->fp8_enc = MCEMU_FP8_FNUZ;
      break;
    case MCEMU_PRESET_CDNA1_FP16: base_desc(out, MCEMU_FP16, MCEMU_ARCH_EXACT, 4); out->nan_bits = 0xFFC00000u; break;
    case MCEMU_PRESET_CDNA1_BF16: base_desc(out, MCEMU_BF16, MCEMU_ARCH_EXACT, 2); out->nan_bits = 0xFFC00000u; break;
    case MCEMU_PRESET_CDNA1_FP32: base_desc(out, MCEMU_FP32, MCEMU_ARCH_EXACT, 1); out->nan_bits = 0xFFC00000u; break;
    case MCEMU_PRESET_CDNA2_FP16: pairwise(out, MCEMU_FP16, 4); break;
    case MCEMU_PRESET_CDNA2_BF16_1K: pairwise(out, MCEMU_BF16, 4); break;
    case MCEMU_PRESET_CDNA2_BF16: pairwise(out, MCEMU_BF16, 2); break;
    case MCEMU_PRESET_B200_FP16: early(out, MCEMU_FP16, 16, 25, MCEMU_OUT_RTZ, -133); break;
    case MCEMU_PRESET_H100_FP16: early(out, MCEMU_FP16, 16, 25, MCEMU_OUT_RTZ, -133); break;
    case MCEMU_PRESET_A100_FP16: early(out, MCEMU_FP16, 8, 24, MCEMU_OUT_RTZ, -132); break;
    case MCEMU_PRESET_B200_BF16: early(out, MCEMU_BF16, 16, 25, MCEMU_OUT_RTZ, -133); break;
    case MCEMU_PRESET_A100_BF16: early(out, MCEMU_BF16, 8, 24, MCEMU_OUT_RTZ, -132); break;
    case MCEMU_PRESET_B200_TF19: early(out, MCEMU_XF32, 8, 25, MCEMU_OUT_RTZ, -133); break;
    case MCEMU_PRESET_A100_TF19: early(out, MCEMU_XF32, 4, 24, MCEMU_OUT_RTZ, -132); break;
    case MCEMU_PRESET_B200_FP8: early(out, MCEMU_E4M3, 32, 25, MCEMU_OUT_RTZ, MCEMU_NO_EXP); break;
    case MCEMU_PRESET_H100_FP8: early(out, MCEMU_E4M3, 32, 13, MCEMU_OUT_RTZ, MCEMU_NO_EXP); break;
    case MCEMU_PRESET_B200_FP16_F16: early16(out, MCEMU_FP16, 16, 25, -21); break;
    case MCEMU_PRESET_H100_FP16_F16: early16(out, MCEMU_FP16, 16, 25, -21); break;
    case MCEMU_PRESET_A100_FP16_F16: early16(out, MCEMU_FP16, 8, 24, -20); break;
    case MCEMU_PRESET_B200_FP8_F16: early16(out, MCEMU_E4M3, 32, 25, -21); break;
    case MCEMU_PRESET_H100_FP8_F16: early16(out, MCEMU_E4M3, 32, 13, -21); break;
    case MCEMU_PRESET_GA_TRUNC:
    case MCEMU_PRESET_GA_RNE:
    case MCEMU_PRESET_IEEE_EXACT: {
      if (fmt < MCEMU_FP16 || fmt > MCEMU_UINT8 || block_k < 1 || block_k > 32) return MCEMU_ERR_INVALID_ARG;
      if (fmt == MCEMU_INT8 || fmt == MCEMU_UINT8) {
        base_desc(out, fmt, MCEMU_ARCH_EXACT, block_k);
      } else if (preset == MCEMU_PRESET_IEEE_EXACT) {
        base_desc(out, fmt, MCEMU_ARCH_EXACT, block_k);
      } else {
        // F_p = 23 + 3 extra alignment bits, truncated alignment, c = 0 discarded
        early(out, fmt, block_k, 26, preset == MCEMU_PRESET_GA_TRUNC ? MCEMU_OUT_RTZ : MCEMU_OUT_RNE,
              MCEMU_NO_EXP);
      }
      break;
    }
    default: return MCEMU_ERR_INVALID_ARG;
  }
  return MCEMU_OK;
}

// ---------------------------------------------------------------------------
// model validation and the kernel-side description
// ---------------------------------------------------------------------------
static bool is_int_fmt(int f) { return f == MCEMU_INT8 || f == MCEMU_UINT8; }

static FmtDev make_fmt(int fmt, int enc, int xr, bool flush) {
  FmtDev f;
  std::memset(&f, 0, sizeof f);
  f.nan_mask = 0u;
  f.nan_pat = 0xFFFFFFFFu;           // "no extra NaN encoding"
  f.top_special = 0xFFFFFFFFu;
  auto ieee = [&](uint32_t e, uint32_t m, int bias) {
    f.mbits = m; f.emask = (1u << e) - 1u; f.sshift = e + m; f.bias = bias;
    f.top_special = (1u << e) - 1u; f.m_eff = (int32_t)m;
    f.sub_keep = flush ? 0u : (1u << m) - 1u;
  };
  switch (fmt) {
    case MCEMU_FP16:
      ieee(5, 10, 15);
      f.sw_mask = 0x7C007C00u; f.sw_add = 0x04000400u; f.sw_hi = 0x80008000u;
      break;
    case MCEMU_BF16:
      ieee(8, 7, 127);
      f.sw_mask = 0x7F807F80u; f.sw_add = 0x00800080u; f.sw_hi = 0x80008000u;
      break;
    case MCEMU_FP32:
    case MCEMU_XF32:
      ieee(8, 23, 127);
      f.sw_mask = 0x7F800000u; f.sw_add = 0x00800000u; f.sw_hi = 0x80000000u;
      if (fmt == MCEMU_XF32) {
        f.xf32 = xr == MCEMU_XF32_RNE ? 2u : 1u;
        f.sig_rshift = 13;
        f.m_eff = 10;
      }
      break;
    case MCEMU_E4M3:
      f.mbits = 3; f.emask = 0xFu; f.sshift = 7; f.m_eff = 3;
      f.sub_keep = flush ? 0u : 7u;
      if (enc == MCEMU_FP8_FNUZ) {
        f.bias = 8; f.nan_mask = 0xFFu; f.nan_pat = 0x80u; f.sw_fnuz = 1;
      } else {
        f.bias = 7; f.nan_mask = 0x7Fu; f.nan_pat = 0x7Fu;   // S.1111.111
        f.sw_mask = 0x7F7F7F7Fu; f.sw_add = 0x01010101u; f.sw_hi = 0x80808080u;
      }
      break;
    case MCEMU_E5M2:
      if (enc == MCEMU_FP8_FNUZ) {
        f.mbits = 2; f.emask = 0x1Fu; f.sshift = 7; f.bias = 16; f.m_eff = 2;
        f.sub_keep = flush ? 0u : 3u;
        f.nan_mask = 0xFFu; f.nan_pat = 0x80u; f.sw_fnuz = 1;
      } else {
        ieee(5, 2, 15);
        f.sw_mask = 0x7C7C7C7Cu; f.sw_add = 0x04040404u; f.sw_hi = 0x80808080u;
      }
      break;
    case MCEMU_INT8:
    case MCEMU_UINT8:
      f.is_int = 1; f.is_signed = fmt == MCEMU_INT8; f.sshift = 7;
      break;
  }
  return f;
}

static bool can_overflow_2p128(int fmt) {
  return fmt == MCEMU_BF16 || fmt == MCEMU_XF32 || fmt == MCEMU_FP32;
}

static int validate(const mcemu_model_desc *d) {
  if (d->struct_size != sizeof(mcemu_model_desc)) return MCEMU_ERR_INVALID_ARG;
  if (d->fmt_a < MCEMU_FP16 || d->fmt_a > MCEMU_UINT8 || d->fmt_b < MCEMU_FP16 || d->fmt_b > MCEMU_UINT8)
    return MCEMU_ERR_INVALID_ARG;
  if (is_int_fmt(d->fmt_a) != is_int_fmt(d->fmt_b)) return MCEMU_ERR_INVALID_ARG;
  if (d->block_k < 1 || d->block_k > 32) return MCEMU_ERR_INVALID_ARG;
  if ((d->int_saturate | 1) != 1 || (d->subnormal_in_flush | 1) != 1 || (d->subnormal_out_flush | 1) != 1)
    return MCEMU_ERR_INVALID_ARG;
  if (is_int_fmt(d->fmt_a)) return MCEMU_OK;
  // one element container size for a and b (the kernels load both the same way)
  auto bytes = [](int f) { return f == MCEMU_FP16 || f == MCEMU_BF16 ? 2 : (f == MCEMU_XF32 || f == MCEMU_FP32 ? 4 : 1); };
  if (bytes(d->fmt_a) != bytes(d->fmt_b)) return MCEMU_ERR_UNSUPPORTED;
  if (d->arch < MCEMU_ARCH_EXACT || d->arch > MCEMU_ARCH_PAIRWISE) return MCEMU_ERR_INVALID_ARG;
  if (d->fp8_enc != MCEMU_FP8_OCP && d->fp8_enc != MCEMU_FP8_FNUZ) return MCEMU_ERR_INVALID_ARG;
  if (d->xf32_round != MCEMU_XF32_TRUNC && d->xf32_round != MCEMU_XF32_RNE) return MCEMU_ERR_INVALID_ARG;
  if (d->out_round != MCEMU_OUT_RNE && d->out_round != MCEMU_OUT_RTZ) return MCEMU_ERR_INVALID_ARG;
  if (d->align_round != MCEMU_ALIGN_RZ && d->align_round != MCEMU_ALIGN_RD) return MCEMU_ERR_INVALID_ARG;
  if (d->acc_sig_bits != 24 && d->acc_sig_bits != 11) return MCEMU_ERR_UNSUPPORTED;
  if (d->acc_sig_bits == 11) {
    // binary16 accumulator: the early-c and exact adders with FP16/FP8 inputs, whose
    // exact sums sit on the 2^-48 grid of the binary16 evaluator
    if (d->arch != MCEMU_ARCH_GA_EARLY && d->arch != MCEMU_ARCH_EXACT) return MCEMU_ERR_UNSUPPORTED;
    auto narrow = [](int f) { return f == MCEMU_FP16 || f == MCEMU_E4M3 || f == MCEMU_E5M2; };
    if (!narrow(d->fmt_a) || !narrow(d->fmt_b)) return MCEMU_ERR_UNSUPPORTED;
    if (d->nan_bits > 0xFFFFu) return MCEMU_ERR_INVALID_ARG;
    // the alignment grid stays below 2^(40 - F_p) (the evaluator's 128-bit terms)
    if (d->emin_lim != MCEMU_NO_EXP && (d->emin_lim < -200 || d->emin_lim > 40)) return MCEMU_ERR_UNSUPPORTED;
    if (d->c_zero_exp != MCEMU_NO_EXP && (d->c_zero_exp < -200 || d->c_zero_exp > 40)) return MCEMU_ERR_UNSUPPORTED;
  }
  if (d->c_zero_exp != MCEMU_NO_EXP && (d->c_zero_exp < -1000 || d->c_zero_exp > 1000)) return MCEMU_ERR_INVALID_ARG;
  if (d->emin_lim != MCEMU_NO_EXP && (d->emin_lim < -1000 || d->emin_lim > 1000)) return MCEMU_ERR_INVALID_ARG;
  if (d->arch == MCEMU_ARCH_GA_EARLY || d->arch == MCEMU_ARCH_GA_LATE || d->arch == MCEMU_ARCH_ODD_EVEN) {
    if (d->align_frac_bits < 0 || d->align_frac_bits > 52) return MCEMU_ERR_UNSUPPORTED;
  }
  if (d->arch == MCEMU_ARCH_GA_LATE || d->arch == MCEMU_ARCH_ODD_EVEN) {
    // 64-bit late-c merge: the shifted product sum stays below 2^(F_p + 7 + (psum - F_p))
    if (d->align_frac_bits > 30) return MCEMU_ERR_UNSUPPORTED;
    if (d->c_frac_bits != d->align_frac_bits) return MCEMU_ERR_UNSUPPORTED;
    if (d->psum_frac_bits < 23 || d->psum_frac_bits < d->align_frac_bits ||
        d->psum_frac_bits > d->align_frac_bits + 8)
      return MCEMU_ERR_UNSUPPORTED;
    if (d->post_norm_frac_bits < 0 || d->post_norm_frac_bits > 60) return MCEMU_ERR_UNSUPPORTED;
    if (d->emin_lim != MCEMU_NO_EXP) return MCEMU_ERR_UNSUPPORTED;
  }
  if (d->arch == MCEMU_ARCH_PAIRWISE) {
    if (d->pair_group != d->block_k) return MCEMU_ERR_UNSUPPORTED;
    if (d->subnormal_in_flush != d->subnormal_out_flush) return MCEMU_ERR_UNSUPPORTED;
    if (d->out_round != MCEMU_OUT_RNE) return MCEMU_ERR_UNSUPPORTED;
  }
  return MCEMU_OK;
}

static DevModel derive(const mcemu_model_desc *d) {
  DevModel m;
  std::memset(&m, 0, sizeof m);
  const bool flush = d->subnormal_in_flush != 0;
  m.fa = make_fmt(d->fmt_a, d->fp8_enc, d->xf32_round, flush);
  m.fb = make_fmt(d->fmt_b, d->fp8_enc, d->xf32_round, flush);
  m.arch = d->arch;
  m.k = d->block_k;
  m.F = d->align_frac_bits;
  m.align_rd = d->align_round == MCEMU_ALIGN_RD;
  m.c_frac = d->c_frac_bits;
  m.psum_frac = d->psum_frac_bits;
  m.post_norm_frac = d->post_norm_frac_bits;
  m.rne = d->out_round == MCEMU_OUT_RNE;
  m.sub_out_flush = d->subnormal_out_flush;
  m.acc16 = d->acc_sig_bits == 11;
  m.c_sub_keep = flush ? 0u : (m.acc16 ? 0x3FFu : 0x7FFFFFu);
  m.c_zero_exp = d->c_zero_exp == MCEMU_NO_EXP ? kNegE : d->c_zero_exp;
  m.emin_lim = d->emin_lim == MCEMU_NO_EXP ? kNegE : d->emin_lim;
  m.prod_ovf = d->prod_overflow_2p128 && (can_overflow_2p128(d->fmt_a) || can_overflow_2p128(d->fmt_b));
  m.nan_bits = d->nan_bits;
  m.int_sat = d->int_saturate;
  m.mab = m.fa.m_eff + m.fb.m_eff;
  int L0 = m.F - m.mab;
  m.P0 = L0 > 0 ? L0 : 0;
  m.R0 = L0 < 0 ? -L0 : 0;
  int L0c = m.F - 23;
  m.P0c = L0c > 0 ? L0c : 0;
  m.R0c = L0c < 0 ? -L0c : 0;
  m.bias_sum = m.fa.bias + m.fb.bias;
  // 32-bit sums: every aligned product is at most (2^(ma+1)-1)(2^(mb+1)-1) << P0 and c
  // at most (2^24-1) << P0c; k of the first plus one c must stay below 2^31
  double pmax = (double)((1ll << (m.fa.m_eff + 1)) - 1) * (double)((1ll << (m.fb.m_eff + 1)) - 1) *
                (double)(1ll << (m.P0 < 40 ? m.P0 : 40));
  double cmax = (double)((1ll << 24) - 1) * (double)(1ll << (m.P0c < 40 ? m.P0c : 40));
  double bound = (double)m.k * pmax + cmax;
  m.wide = (m.F + 2 > 31) || (m.mab > 22) || bound >= 2147483648.0;
  m.p0mul = m.P0 < 32 ? 1u << m.P0 : 0u;
  m.p0cmul = m.P0c < 32 ? 1u << m.P0c : 0u;
  return m;
}

extern "C" int mcemu_model_create(const mcemu_model_desc *desc, mcemu_model_t *out) {
  if (!desc || !out) return MCEMU_ERR_INVALID_ARG;
  *out = nullptr;
  int st = validate(desc);
  if (st != MCEMU_OK) return st;
  mcemu_model *h = new (std::nothrow) mcemu_model;
  if (!h) return MCEMU_ERR_INVALID_ARG;
  h->m.desc = *desc;
  h->m.dev = derive(desc);
  *out = h;
  return MCEMU_OK;
}

extern "C" void mcemu_model_destroy(mcemu_model_t model) { delete model; }

extern "C" int mcemu_model_get_desc(mcemu_model_t model, mcemu_model_desc *out) {
  if (!model || !out) return MCEMU_ERR_INVALID_ARG;
  *out = model->m.desc;
  return MCEMU_OK;
}

// ---------------------------------------------------------------------------
// block-FMA stream
// ---------------------------------------------------------------------------
static int elem_bytes(int fmt) {
  return fmt == MCEMU_FP16 || fmt == MCEMU_BF16 ? 2 : (fmt == MCEMU_XF32 || fmt == MCEMU_FP32 ? 4 : 1);
}

static bool aligned(const void *p, size_t a) { return ((uintptr_t)p % a) == 0; }

extern "C" int mcemu_block_fma(mcemu_model_t model, size_t n, const void *a, const void *b,
                               const uint32_t *c, uint32_t *d, void *stream) {
  if (!model) return MCEMU_ERR_INVALID_ARG;
  if (n == 0) return MCEMU_OK;
  if (!a || !b || !c || !d) return MCEMU_ERR_INVALID_ARG;
  const DevModel &m = model->m.dev;
  const size_t eb = elem_bytes(model->m.desc.fmt_a), vec = (size_t)m.k * eb;
  // vector sets of a power-of-two size are loaded whole (up to 16 bytes at a time);
  // other sizes element by element
  const size_t need = (vec & (vec - 1)) == 0 ? (vec < 16 ? vec : 16) : eb;
  if (!aligned(a, need) || !aligned(b, need) || !aligned(c, 4) || !aligned(d, 4)) return MCEMU_ERR_ALIGNMENT;
  return launch_block_fma(m, n, a, b, c, d, stream);
}

// Host buffers: chunks of the vector sets are copied into the caller's device
// workspace and processed, two chunk buffers alternating so that the copies of
// one chunk overlap the kernel of the other (one stream per buffer, events
// keep the order).
static const size_t kHostChunk = (size_t)1 << 22;   // vectors per chunk

extern "C" size_t mcemu_block_fma_host_workspace(mcemu_model_t model) {
  if (!model) return 0;
  size_t vec = (size_t)model->m.dev.k * elem_bytes(model->m.desc.fmt_a);
  size_t per = 2 * ((vec * kHostChunk + 255) & ~(size_t)255) + 2 * ((4 * kHostChunk + 255) & ~(size_t)255);
  return 2 * per;
}

// a host pointer the device can dereference as it is: page-locked host memory mapped into
// the unified address space (the device pointer equals the host pointer)
static bool host_mapped(const void *p) {
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();                                // an unregistered pointer, on older runtimes
    return false;
  }
  return at.type == cudaMemoryTypeHost && at.devicePointer == p;
}

extern "C" int mcemu_block_fma_host(mcemu_model_t model, size_t n, const void *a, const void *b,
                                    const uint32_t *c, uint32_t *d, void *workspace, size_t ws_bytes,
                                    void *stream) {
  if (!model) return MCEMU_ERR_INVALID_ARG;
  if (n == 0) return MCEMU_OK;
  if (!a || !b || !c || !d || !workspace) return MCEMU_ERR_INVALID_ARG;
  if (ws_bytes < mcemu_block_fma_host_workspace(model)) return MCEMU_ERR_WORKSPACE;
  if (!aligned(workspace, 256)) return MCEMU_ERR_ALIGNMENT;
  const DevModel &m = model->m.dev;
  const size_t vec = (size_t)m.k * elem_bytes(model->m.desc.fmt_a);
  cudaStream_t s0 = (cudaStream_t)stream;
  // page-locked buffers mapped into the device's address space: the kernels stream them
  // in place over the host link, which beats staging through the copy engines
  if (host_mapped(a) && host_mapped(b) && host_mapped(c) && host_mapped(d)) {
    const int st = launch_block_fma(m, n, a, b, c, d, s0);
    if (st != MCEMU_OK) return st;
    return cudaStreamSynchronize(s0) == cudaSuccess ? MCEMU_OK : MCEMU_ERR_CUDA;
  }
  const size_t sa = (vec * kHostChunk + 255) & ~(size_t)255, sc = (4 * kHostChunk + 255) & ~(size_t)255;
  cudaStream_t ss[2];
  cudaEvent_t done[2];
  if (cudaStreamCreateWithFlags(&ss[0], cudaStreamNonBlocking) != cudaSuccess) return MCEMU_ERR_CUDA;
  if (cudaStreamCreateWithFlags(&ss[1], cudaStreamNonBlocking) != cudaSuccess) {
    cudaStreamDestroy(ss[0]);
    return MCEMU_ERR_CUDA;
  }
  cudaEventCreateWithFlags(&done[0], cudaEventDisableTiming);
  cudaEventCreateWithFlags(&done[1], cudaEventDisableTiming);
  // both workers start after work already queued on the caller's stream
  cudaEventRecord(done[0], s0);
  cudaStreamWaitEvent(ss[0], done[0], 0);
  cudaStreamWaitEvent(ss[1], done[0], 0);
  int st = MCEMU_OK;
  uint8_t *ws = (uint8_t *)workspace;
  for (size_t off = 0, it = 0; off < n && st == MCEMU_OK; off += kHostChunk, it++) {
    const int w = (int)(it & 1);
    cudaStream_t s = ss[w];
    uint8_t *base = ws + w * (2 * sa + 2 * sc);
    uint8_t *da = base, *db = base + sa;
    uint32_t *dc = (uint32_t *)(base + 2 * sa), *dd = (uint32_t *)(base + 2 * sa + sc);
    const size_t cnt = (n - off < kHostChunk) ? n - off : kHostChunk;
    if (cudaMemcpyAsync(da, (const uint8_t *)a + off * vec, cnt * vec, cudaMemcpyHostToDevice, s) != cudaSuccess ||
        cudaMemcpyAsync(db, (const uint8_t *)b + off * vec, cnt * vec, cudaMemcpyHostToDevice, s) != cudaSuccess ||
        cudaMemcpyAsync(dc, c + off, cnt * 4, cudaMemcpyHostToDevice, s) != cudaSuccess) {
      st = MCEMU_ERR_CUDA;
      break;
    }
    st = launch_block_fma(m, cnt, da, db, dc, dd, s);
    if (st != MCEMU_OK) break;
    if (cudaMemcpyAsync(d + off, dd, cnt * 4, cudaMemcpyDeviceToHost, s) != cudaSuccess) st = MCEMU_ERR_CUDA;
  }
  if (cudaStreamSynchronize(ss[0]) != cudaSuccess) st = MCEMU_ERR_CUDA;
  if (cudaStreamSynchronize(ss[1]) != cudaSuccess) st = MCEMU_ERR_CUDA;
  cudaEventDestroy(done[0]);
  cudaEventDestroy(done[1]);
  cudaStreamDestroy(ss[0]);
  cudaStreamDestroy(ss[1]);
  return st;
}

// ---------------------------------------------------------------------------
// tile semantics (CDNA3 dense MFMA page "Accumulator layout"; RDNA4 sparse WMMA
// page "Fragment layouts")
// ---------------------------------------------------------------------------
extern "C" int mcemu_tile_info(const mcemu_tile_desc *t, int32_t *blocks, int32_t *acc_regs) {
  if (!t || !blocks || !acc_regs) return MCEMU_ERR_INVALID_ARG;
  if (t->M <= 0 || t->N <= 0 || t->K <= 0 || t->elems_per_lane <= 0) return MCEMU_ERR_INVALID_ARG;
  if (t->family == 0) {
    int per_wave = 64 * t->elems_per_lane;           // A elements supplied by a wave64
    if (per_wave % (t->M * t->K) != 0) return MCEMU_ERR_INVALID_ARG;
    int b = per_wave / (t->M * t->K);
    if ((b * t->M * t->N) % 64 != 0) return MCEMU_ERR_INVALID_ARG;
    *blocks = b;
    *acc_regs = b * t->M * t->N / 64;
    return MCEMU_OK;
  }
  if (t->family == 1) {
    if (t->M != 16 || t->N != 16) return MCEMU_ERR_UNSUPPORTED;
    *blocks = 1;
    *acc_regs = t->M * t->N / 32;
    return MCEMU_OK;
  }
  return MCEMU_ERR_INVALID_ARG;
}

extern "C" int mcemu_tile_layout(const mcemu_tile_desc *t, int f64, int i, int j, int b,
                                 int32_t *lane, int32_t *reg) {
  if (!t || !lane || !reg) return MCEMU_ERR_INVALID_ARG;
  int32_t blocks = 1, acc = 0;
  if (t->family == 0 && f64) {
    blocks = (t->M == 4) ? 4 : 1;
  } else if (mcemu_tile_info(t, &blocks, &acc) != MCEMU_OK) {
    return MCEMU_ERR_INVALID_ARG;
  }
  if (i < 0 || i >= t->M || j < 0 || j >= t->N || b < 0 || b >= blocks || t->M != t->N)
    return MCEMU_ERR_INVALID_ARG;
  if (t->family == 1) {                       // SWMMAC D: lane = floor(i/8)*16 + j, VGPR = i mod 8
    *lane = (i / 8) * 16 + j;
    *reg = i % 8;
    return MCEMU_OK;
  }
  if (!f64) {
    switch (t->M) {
      case 32: *lane = (32 * (i / 4)) % 64 + j; *reg = 16 * b + 4 * (i / 8) + i % 4; return MCEMU_OK;
      case 16: *lane = 16 * (i / 4) + j; *reg = 4 * b + i % 4; return MCEMU_OK;
      case 4: *lane = 4 * b + j; *reg = i; return MCEMU_OK;
      default: return MCEMU_ERR_UNSUPPORTED;
    }
  }
  switch (t->M) {
    case 16: *lane = 16 * (i % 4) + j; *reg = i / 4; return MCEMU_OK;    // FP64 16x16: pair k
    case 4: *lane = 16 * i + 4 * b + j; *reg = 0; return MCEMU_OK;       // FP64 4x4
    default: return MCEMU_ERR_UNSUPPORTED;
  }
}

extern "C" int mcemu_tile_layout_inverse(const mcemu_tile_desc *t, int f64, int lane, int reg,
                                         int32_t *i, int32_t *j, int32_t *b) {
  if (!t || !i || !j || !b) return MCEMU_ERR_INVALID_ARG;
  if (t->family == 1) {
    if (lane < 0 || lane >= 32 || reg < 0 || reg >= 8) return MCEMU_ERR_INVALID_ARG;
    *i = (lane / 16) * 8 + reg; *j = lane % 16; *b = 0;
    return MCEMU_OK;
  }
  if (lane < 0 || lane >= 64 || reg < 0) return MCEMU_ERR_INVALID_ARG;
  if (!f64) {
    int32_t blocks = 0, acc = 0;
    if (mcemu_tile_info(t, &blocks, &acc) != MCEMU_OK || reg >= acc) return MCEMU_ERR_INVALID_ARG;
    switch (t->M) {
      case 32: *i = (8 * (reg / 4)) % 32 + 4 * (lane / 32) + reg % 4; *j = lane % 32; *b = reg / 16; return MCEMU_OK;
      case 16: *i = 4 * (lane / 16) + reg % 4; *j = lane % 16; *b = reg / 4; return MCEMU_OK;
      case 4: *i = reg % 4; *j = lane % 4; *b = lane / 4; return MCEMU_OK;
      default: return MCEMU_ERR_UNSUPPORTED;
    }
  }
  switch (t->M) {
    case 16: if (reg >= 4) return MCEMU_ERR_INVALID_ARG; *i = 4 * reg + lane / 16; *j = lane % 16; *b = 0; return MCEMU_OK;
    case 4: if (reg != 0) return MCEMU_ERR_INVALID_ARG; *i = lane / 16; *j = lane % 4; *b = (lane % 16) / 4; return MCEMU_OK;
    default: return MCEMU_ERR_UNSUPPORTED;
  }
}

extern "C" int mcemu_swmmac_src_layout(int operand, int idx, int k, int32_t *lane, int32_t *vgpr,
                                       int32_t *half) {
  if (!lane || !vgpr || !half || idx < 0 || idx >= 16) return MCEMU_ERR_INVALID_ARG;
  if (operand == 0) {            // compressed K {0-3, 8-11} in lanes 0-15, {4-7, 12-15} in 16-31
    if (k < 0 || k >= 16) return MCEMU_ERR_INVALID_ARG;
    *lane = 16 * ((k >> 2) & 1) + idx;
    *vgpr = 2 * (k >> 3) + ((k & 3) >> 1);
    *half = k & 1;
    return MCEMU_OK;
  }
  if (operand == 1) {            // dense K rows {0-7, 16-23} in lanes 0-15, {8-15, 24-31} in 16-31
    if (k < 0 || k >= 32) return MCEMU_ERR_INVALID_ARG;
    *lane = 16 * ((k >> 3) & 1) + idx;
    *vgpr = 4 * (k >> 4) + ((k & 7) >> 1);
    *half = k & 1;
    return MCEMU_OK;
  }
  return MCEMU_ERR_INVALID_ARG;
}

// ---------------------------------------------------------------------------
// GEMM entry points
// ---------------------------------------------------------------------------
static int check_tile(const mcemu_tile_desc *t) {
  if (!t || t->K <= 0 || t->M <= 0 || t->N <= 0) return MCEMU_ERR_INVALID_ARG;
  return MCEMU_OK;
}

extern "C" int mcemu_tile_gemm(mcemu_model_t model, const mcemu_tile_desc *tile, int M, int N, int K,
                               const void *A, int64_t lda, const void *Bt, int64_t ldb,
                               const uint32_t *C, int64_t ldc, uint32_t *D, int64_t ldd, void *stream) {
  if (!model || check_tile(tile) != MCEMU_OK) return MCEMU_ERR_INVALID_ARG;
  if (M < 0 || N < 0 || K < 0) return MCEMU_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return MCEMU_OK;
  if (!A && K > 0) return MCEMU_ERR_INVALID_ARG;
  if ((!Bt && K > 0) || !C || !D) return MCEMU_ERR_INVALID_ARG;
  if (lda < K || ldb < K || ldc < N || ldd < N) return MCEMU_ERR_INVALID_ARG;
  if (!aligned(C, 4) || !aligned(D, 4)) return MCEMU_ERR_ALIGNMENT;
  return launch_tile_gemm(model->m.dev, tile->K, M, N, K, A, lda, Bt, ldb, C, ldc, D, ldd, stream);
}

extern "C" int mcemu_sparse24_compress(int fmt, int fp8_enc, int M, int K, const void *A, int64_t lda,
                                       void *Ac, int64_t ldac, uint8_t *meta, int64_t ldm,
                                       int64_t *d_violations, void *stream) {
  if (fmt < MCEMU_FP16 || fmt > MCEMU_UINT8) return MCEMU_ERR_INVALID_ARG;
  if (fp8_enc != MCEMU_FP8_OCP && fp8_enc != MCEMU_FP8_FNUZ) return MCEMU_ERR_INVALID_ARG;
  if (M < 0 || K < 0 || K % 4 != 0) return MCEMU_ERR_INVALID_ARG;
  if (M == 0 || K == 0) return MCEMU_OK;
  if (!A || !Ac || !meta || !d_violations) return MCEMU_ERR_INVALID_ARG;
  if (lda < K || ldac < K / 2 || ldm < K / 4) return MCEMU_ERR_INVALID_ARG;
  if (!aligned(d_violations, 8)) return MCEMU_ERR_ALIGNMENT;
  FmtDev f = make_fmt(fmt, fp8_enc, MCEMU_XF32_TRUNC, false);
  return launch_sparse24_compress(f, elem_bytes(fmt), M, K, A, lda, Ac, ldac, meta, ldm, d_violations, stream);
}

extern "C" int mcemu_sparse24_check(const int64_t *d_violations, int64_t *h_count, void *stream) {
  if (!d_violations) return MCEMU_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  int64_t v = 0;
  if (cudaMemcpyAsync(&v, d_violations, sizeof v, cudaMemcpyDeviceToHost, s) != cudaSuccess) return MCEMU_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return MCEMU_ERR_CUDA;
  if (h_count) *h_count = v;
  return v ? MCEMU_ERR_NOT_2_4 : MCEMU_OK;
}

extern "C" int mcemu_sparse24_expand(int fmt, int M, int K, const void *Ac, int64_t ldac,
                                     const uint8_t *meta, int64_t ldm, void *A, int64_t lda, void *stream) {
  if (fmt < MCEMU_FP16 || fmt > MCEMU_UINT8) return MCEMU_ERR_INVALID_ARG;
  if (M < 0 || K < 0 || K % 4 != 0) return MCEMU_ERR_INVALID_ARG;
  if (M == 0 || K == 0) return MCEMU_OK;
  if (!A || !Ac || !meta) return MCEMU_ERR_INVALID_ARG;
  if (lda < K || ldac < K / 2 || ldm < K / 4) return MCEMU_ERR_INVALID_ARG;
  return launch_sparse24_expand(elem_bytes(fmt), M, K, Ac, ldac, meta, ldm, A, lda, stream);
}

extern "C" int mcemu_sparse24_gemm(mcemu_model_t model, const mcemu_tile_desc *tile, int M, int N, int K,
                                   const void *Ac, int64_t ldac, const uint8_t *meta, int64_t ldm,
                                   const void *Bt, int64_t ldb, const uint32_t *C, int64_t ldc,
                                   uint32_t *D, int64_t ldd, void *stream) {
  if (!model || check_tile(tile) != MCEMU_OK) return MCEMU_ERR_INVALID_ARG;
  if (M < 0 || N < 0 || K < 0 || K % 4 != 0 || tile->K % 4 != 0) return MCEMU_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return MCEMU_OK;
  if ((K > 0 && (!Ac || !meta || !Bt)) || !C || !D) return MCEMU_ERR_INVALID_ARG;
  if (ldac < K / 2 || ldm < K / 4 || ldb < K || ldc < N || ldd < N) return MCEMU_ERR_INVALID_ARG;
  if (!aligned(C, 4) || !aligned(D, 4)) return MCEMU_ERR_ALIGNMENT;
  return launch_sparse24_gemm(model->m.dev, tile->K, M, N, K, Ac, ldac, meta, ldm, Bt, ldb, C, ldc, D,
                              ldd, stream);
}

extern "C" int mcemu_multiword_split(int n_words, size_t n, const double *x, uint16_t *words, void *stream) {
  if (n_words < 1 || n_words > 8) return MCEMU_ERR_INVALID_ARG;
  if (n == 0) return MCEMU_OK;
  if (!x || !words) return MCEMU_ERR_INVALID_ARG;
  if (!aligned(x, 8) || !aligned(words, 2)) return MCEMU_ERR_ALIGNMENT;
  return launch_multiword_split(n_words, n, x, (int64_t)n, 1, words, (int64_t)n, stream);
}

extern "C" size_t mcemu_multiword_workspace(int n_words, int M, int N, int K) {
  if (n_words < 1 || n_words > 8 || M < 0 || N < 0 || K < 0) return 0;
  size_t wa = ((size_t)n_words * M * K * 2 + 255) & ~(size_t)255;
  size_t wb = ((size_t)n_words * N * K * 2 + 255) & ~(size_t)255;
  size_t wp = ((size_t)M * N * 4 + 255) & ~(size_t)255;       // one fp32 word product
  return wa + wb + wp;
}

extern "C" int mcemu_multiword_gemm(mcemu_model_t word_model, const mcemu_tile_desc *tile, int n_words,
                                    int product_set, int M, int N, int K, const double *A, int64_t lda,
                                    const double *Bt, int64_t ldb, double *D, int64_t ldd,
                                    void *workspace, size_t ws_bytes, void *stream) {
  if (!word_model || check_tile(tile) != MCEMU_OK) return MCEMU_ERR_INVALID_ARG;
  const mcemu_model_desc &wd = word_model->m.desc;
  if (wd.fmt_a != MCEMU_BF16 || wd.fmt_b != MCEMU_BF16) return MCEMU_ERR_UNSUPPORTED;
  if (n_words < 1 || n_words > 8) return MCEMU_ERR_INVALID_ARG;
  if (product_set != MCEMU_WORDS_ALL && product_set != MCEMU_WORDS_TRUNCATED) return MCEMU_ERR_INVALID_ARG;
  if (M < 0 || N < 0 || K < 0) return MCEMU_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return MCEMU_OK;
  if ((K > 0 && (!A || !Bt)) || !D) return MCEMU_ERR_INVALID_ARG;
  if (lda < K || ldb < K || ldd < N) return MCEMU_ERR_INVALID_ARG;
  if (ws_bytes < mcemu_multiword_workspace(n_words, M, N, K)) return MCEMU_ERR_WORKSPACE;
  if (!workspace || !aligned(workspace, 256)) return workspace ? MCEMU_ERR_ALIGNMENT : MCEMU_ERR_INVALID_ARG;
  if (!aligned(A, 8) || !aligned(Bt, 8) || !aligned(D, 8)) return MCEMU_ERR_ALIGNMENT;
  return launch_multiword_gemm(word_model->m.dev, tile->K, n_words, product_set == MCEMU_WORDS_TRUNCATED, M,
                               N, K, A, lda, Bt, ldb, D, ldd, workspace, ws_bytes, stream);
}

extern "C" int mcemu_multiword_gemm_static(mcemu_model_t word_model, const mcemu_tile_desc *tile, int n_words,
                                           int product_set, int M, int N, int K, const double *A, int64_t lda,
                                           const double *Bt, int64_t ldb, double *D, int64_t ldd, void *stream) {
  if (!word_model || check_tile(tile) != MCEMU_OK) return MCEMU_ERR_INVALID_ARG;
  const mcemu_model_desc &wd = word_model->m.desc;
  if (wd.fmt_a != MCEMU_BF16 || wd.fmt_b != MCEMU_BF16) return MCEMU_ERR_UNSUPPORTED;
  if (n_words < 1 || n_words > 8) return MCEMU_ERR_INVALID_ARG;
  if (product_set != MCEMU_WORDS_ALL && product_set != MCEMU_WORDS_TRUNCATED) return MCEMU_ERR_INVALID_ARG;
  if (M < 0 || N < 0 || K < 0) return MCEMU_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return MCEMU_OK;
  // the words must fit the fixed array (M*K and N*K first, so the size cannot wrap)
  if ((uint64_t)M * (uint64_t)K > MCEMU_MULTIWORD_STATIC_BYTES ||
      (uint64_t)N * (uint64_t)K > MCEMU_MULTIWORD_STATIC_BYTES ||
      mcemu_multiword_workspace(n_words, M, N, K) > MCEMU_MULTIWORD_STATIC_BYTES)
    return MCEMU_ERR_WORKSPACE;
  if ((K > 0 && (!A || !Bt)) || !D) return MCEMU_ERR_INVALID_ARG;
  if (lda < K || ldb < K || ldd < N) return MCEMU_ERR_INVALID_ARG;
  if (!aligned(A, 8) || !aligned(Bt, 8) || !aligned(D, 8)) return MCEMU_ERR_ALIGNMENT;
  return launch_multiword_gemm_static(word_model->m.dev, tile->K, n_words, product_set == MCEMU_WORDS_TRUNCATED,
                                      M, N, K, A, lda, Bt, ldb, D, ldd, stream);
}

extern "C" int mcemu_fro_error(int M, int N, const double *D, int64_t ldd, const double *R, int64_t ldr,
                               double *out, void *stream) {
  if (M < 0 || N < 0 || !out) return MCEMU_ERR_INVALID_ARG;
  if (M > 0 && N > 0 && (!D || !R || ldd < N || ldr < N)) return MCEMU_ERR_INVALID_ARG;
  return launch_fro_error(M, N, D, ldd, R, ldr, out, stream);
}
