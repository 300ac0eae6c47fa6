// kda_chunk_ffma.cu -- chunk-wise gated delta rule on CUDA cores, float32.
//
// The general path: every supported shape (dk, dv in {16,32,64,128},
// C in {16,32,64}), both storage types, any T.  It is the only path for
// float32 inputs, whose tolerance bf16 tensor-core operands cannot meet.
//
// One CTA per (batch*head, block of <= 32 value columns).  The value columns
// of S never mix in the recurrence (W, T and the masks depend only on k,
// beta and the decay), so the blocks are independent; each recomputes the
// key-side quantities of every chunk.  Per chunk of C tokens, with g the
// running sum of log(a) = -exp(log_alpha) from the chunk start and
// gamma = exp(g), gamma_C its value at the chunk end:
//   Kg = K*gamma, Kh = K/gamma, Qg = Q*gamma                     (decayed tiles)
//   A  = strict_lower(diag(beta) Kg Kh^T),  M = lower_incl(Qg Kh^T)
//   [W | U] = (I + A)^-1 [diag(beta) Kg | diag(beta) V]   (forward substitution)
//   u = U - W S;   o = Qg S + M u;   S = Diag(gamma_C) (S + Kh^T u)
// (the tiles are kept relative to gamma at mid-chunk; see step 1)
// With no decay this is the chunked DeltaNet loop of "22,580: From GPT-2 to
// Kimi K3" (yichencityu.github.io), section 6.3 (forward substitution on the
// C x C unit lower-triangular matrix, W = T K_beta, U = T V_beta, then
// u = U - W S, o = q S + tril(q k^T) u, S += k^T u); the decay factors carry
// the cumulative products the gated form needs ("22580: From GPT-2 to
// Kimi3, Explained" (zharfai.com), "Gated DeltaNet adds controlled
// forgetting").  Here (I + A) is solved directly against the right-hand
// sides, which is the same forward substitution without forming T.
//
// A partial last chunk is padded with k = q = v = 0, beta = 0 and a = 1:
// such rows add nothing to A, W, U or u and leave the decay unchanged.
#include "kda_launch.cuh"

namespace kda {
namespace {

constexpr int kFfmaThreads = 256;
constexpr int kMaxDvBlock = 32;

template <int DK>
struct FfmaSmem {
  static constexpr int LDK = DK + 1;  // padded row stride (bank-conflict free)
  static size_t floats(int C, int DVB) {
    const int LDC = C + 1, LDV = DVB + 1;
    return (size_t)4 * C * LDK + (size_t)2 * C * LDC + (size_t)2 * C * LDV +
           (size_t)DK * LDV + 3 * DK + C;
  }
};

template <int DK, typename TI>
__global__ void __launch_bounds__(kFfmaThreads)
chunk_ffma_kernel(const TI *__restrict__ q, const TI *__restrict__ k,
                  const TI *__restrict__ v, const float *__restrict__ beta,
                  const float *__restrict__ log_alpha, int alpha_mode,
                  const float *h0, TI *__restrict__ o, float *hT, int T, int dv,
                  int C, int DVB) {
  constexpr int LDK = FfmaSmem<DK>::LDK;
  const int LDC = C + 1, LDV = DVB + 1;
  extern __shared__ float smem[];
  float *Kg = smem;                 // [C][LDK]  K * gamma
  float *Kh = Kg + C * LDK;         // [C][LDK]  K / gamma
  float *Qg = Kh + C * LDK;         // [C][LDK]  Q * gamma
  float *Wm = Qg + C * LDK;         // [C][LDK]  beta Kg, then W
  float *Am = Wm + C * LDK;         // [C][LDC]  strict lower A
  float *Mm = Am + C * LDC;         // [C][LDC]  inclusive lower M
  float *Ub = Mm + C * LDC;         // [C][LDV]  beta V, then U
  float *Vu = Ub + C * LDV;         // [C][LDV]  V, then u
  float *Sm = Vu + C * LDV;         // [DK][LDV] state block
  float *gC = Sm + DK * LDV;        // [DK]      gamma at chunk end
  float *gCm = gC + DK;             // [DK]      gamma at chunk end / gamma at mid-chunk
  float *em = gCm + DK;             // [DK]      gamma at mid-chunk
  float *bet = em + DK;             // [C]       beta (0 on padded rows)

  const int tid = threadIdx.x;
  const int bh = blockIdx.y;
  const int j0 = blockIdx.x * DVB;
  const size_t qk_base = (size_t)bh * T * DK;
  const size_t v_base = (size_t)bh * T * dv;
  const size_t s_base = (size_t)bh * DK * dv;

  for (int idx = tid; idx < DK * DVB; idx += kFfmaThreads) {
    const int c = idx / DVB, j = idx % DVB;
    Sm[c * LDV + j] = h0 ? h0[s_base + (size_t)c * dv + j0 + j] : 0.f;
  }

  const int NC = (T + C - 1) / C;
  for (int n = 0; n < NC; ++n) {
    const int t0 = n * C;
    const int valid = min(C, T - t0);
    __syncthreads();  // previous chunk finished with every tile

    // (1) decay prefix in log space, decayed tiles; one thread per key channel.
    // The tiles carry gamma relative to its value m at the middle of the chunk
    // (the split factors e^(g-m), e^(m-g) stay within the half chunk's decay,
    // so they stay finite up to about e^87 per half chunk); A and M only see
    // ratios, and the chunk-start values are restored where they are needed.
    if (tid < DK) {
      const int c = tid;
      auto ld_of = [&](int r) -> float {
        if (r >= valid) return 0.f;
        if (alpha_mode == KDA_ALPHA_CHANNEL)
          return log_decay_of(log_alpha[qk_base + (size_t)(t0 + r) * DK + c]);
        if (alpha_mode == KDA_ALPHA_SCALAR) return log_decay_of(log_alpha[(size_t)bh * T + t0 + r]);
        return 0.f;
      };
      float mid = 0.f;
      for (int r = 0; r < C / 2; ++r) mid += ld_of(r);
      float acc = -mid;
      for (int r = 0; r < C; ++r) {
        float kv = 0.f, qv = 0.f;
        if (r < valid) {
          const size_t e = qk_base + (size_t)(t0 + r) * DK + c;
          kv = Io<TI>::ld(k + e);
          qv = Io<TI>::ld(q + e);
        }
        acc += ld_of(r);
        const float gm = expf(acc), gi = expf(-acc);
        Kg[r * LDK + c] = kv * gm;
        Kh[r * LDK + c] = kv * gi;
        Qg[r * LDK + c] = qv * gm;
      }
      gC[c] = expf(acc + mid);
      gCm[c] = expf(acc);
      em[c] = expf(mid);
    }
    for (int r = tid; r < C; r += kFfmaThreads)
      bet[r] = (r < valid) ? beta[(size_t)bh * T + t0 + r] : 0.f;
    for (int idx = tid; idx < C * DVB; idx += kFfmaThreads) {
      const int r = idx / DVB, j = idx % DVB;
      Vu[r * LDV + j] = (r < valid) ? Io<TI>::ld(v + v_base + (size_t)(t0 + r) * dv + j0 + j) : 0.f;
    }
    __syncthreads();

    // (2) A = strict_lower(diag(beta) Kg Kh^T), M = lower_incl(Qg Kh^T);
    // (3) right-hand sides beta Kg and beta V.
    for (int idx = tid; idx < C * C; idx += kFfmaThreads) {
      const int r = idx / C, j = idx % C;
      float a = 0.f, m = 0.f;
      if (j <= r) {
        const float *kr = Kg + r * LDK, *qr = Qg + r * LDK, *kj = Kh + j * LDK;
        for (int c = 0; c < DK; ++c) {
          a += kr[c] * kj[c];
          m += qr[c] * kj[c];
        }
      }
      Am[r * LDC + j] = (j < r) ? bet[r] * a : 0.f;
      Mm[r * LDC + j] = m;
    }
    for (int idx = tid; idx < C * DK; idx += kFfmaThreads) {
      const int r = idx / DK, c = idx % DK;
      Wm[r * LDK + c] = bet[r] * Kg[r * LDK + c] * em[c];  // beta K gamma, chunk-start gamma
    }
    for (int idx = tid; idx < C * DVB; idx += kFfmaThreads) {
      const int r = idx / DVB, j = idx % DVB;
      Ub[r * LDV + j] = bet[r] * Vu[r * LDV + j];
    }
    __syncthreads();

    // (4) forward substitution: row i of [W | U] minus A[i, :i] times the
    // finished rows above it.
    for (int i = 1; i < C; ++i) {
      for (int col = tid; col < DK + DVB; col += kFfmaThreads) {
        const float *ai = Am + i * LDC;
        if (col < DK) {
          float x = Wm[i * LDK + col];
          for (int m = 0; m < i; ++m) x -= ai[m] * Wm[m * LDK + col];
          Wm[i * LDK + col] = x;
        } else {
          const int j = col - DK;
          float x = Ub[i * LDV + j];
          for (int m = 0; m < i; ++m) x -= ai[m] * Ub[m * LDV + j];
          Ub[i * LDV + j] = x;
        }
      }
      __syncthreads();
    }

    // (5) u = U - W S  (into Vu)
    for (int idx = tid; idx < C * DVB; idx += kFfmaThreads) {
      const int r = idx / DVB, j = idx % DVB;
      float acc = Ub[r * LDV + j];
      const float *wr = Wm + r * LDK;
      for (int c = 0; c < DK; ++c) acc -= wr[c] * Sm[c * LDV + j];
      Vu[r * LDV + j] = acc;
    }
    __syncthreads();

    // (6) o = Qg S + M u  (rows of the chunk that exist)
    for (int idx = tid; idx < C * DVB; idx += kFfmaThreads) {
      const int r = idx / DVB, j = idx % DVB;
      if (r < valid) {
        float acc = 0.f;
        const float *qr = Qg + r * LDK;
        for (int c = 0; c < DK; ++c) acc += qr[c] * em[c] * Sm[c * LDV + j];
        const float *mr = Mm + r * LDC;
        for (int m = 0; m <= r; ++m) acc += mr[m] * Vu[m * LDV + j];
        Io<TI>::st(o + v_base + (size_t)(t0 + r) * dv + j0 + j, acc);
      }
    }
    __syncthreads();

    // (7) S = Diag(gamma_C) S + Kbar^T u, Kbar = K gamma_C / gamma = Kh gamma_C / gamma_mid
    for (int idx = tid; idx < DK * DVB; idx += kFfmaThreads) {
      const int c = idx / DVB, j = idx % DVB;
      float acc = 0.f;
      for (int r = 0; r < C; ++r) acc += Kh[r * LDK + c] * Vu[r * LDV + j];
      Sm[c * LDV + j] = gC[c] * Sm[c * LDV + j] + gCm[c] * acc;
    }
  }
  __syncthreads();
  if (hT) {
    for (int idx = tid; idx < DK * DVB; idx += kFfmaThreads) {
      const int c = idx / DVB, j = idx % DVB;
      hT[s_base + (size_t)c * dv + j0 + j] = Sm[c * LDV + j];
    }
  }
}

template <int DK, typename TI>
kda_status launch_ffma_t(const void *q, const void *k, const void *v, const float *beta,
                         const float *la, const float *h0, void *o, float *hT, int BH,
                         int T, int dv, int C, int am, cudaStream_t st, LaunchTimer &timer) {
  const int DVB = dv < kMaxDvBlock ? dv : kMaxDvBlock;
  const size_t smem = FfmaSmem<DK>::floats(C, DVB) * sizeof(float);
  auto kern = chunk_ffma_kernel<DK, TI>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
      cudaSuccess)
    return KDA_ERR_CUDA;
  const dim3 grid(dv / DVB, BH), block(kFfmaThreads);
  timer.mark();
  kern<<<grid, block, smem, st>>>(static_cast<const TI *>(q), static_cast<const TI *>(k),
                                  static_cast<const TI *>(v), beta, la, am, h0,
                                  static_cast<TI *>(o), hT, T, dv, C, DVB);
  timer.mark();
  return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

template <typename TI>
kda_status launch_ffma_dt(const void *q, const void *k, const void *v, const float *beta,
                          const float *la, const float *h0, void *o, float *hT, int BH, int T,
                          int dk, int dv, int C, int am, cudaStream_t st, LaunchTimer &tm) {
  switch (dk) {
    case 16: return launch_ffma_t<16, TI>(q, k, v, beta, la, h0, o, hT, BH, T, dv, C, am, st, tm);
    case 32: return launch_ffma_t<32, TI>(q, k, v, beta, la, h0, o, hT, BH, T, dv, C, am, st, tm);
    case 64: return launch_ffma_t<64, TI>(q, k, v, beta, la, h0, o, hT, BH, T, dv, C, am, st, tm);
    case 128: return launch_ffma_t<128, TI>(q, k, v, beta, la, h0, o, hT, BH, T, dv, C, am, st, tm);
    default: return KDA_ERR_UNSUPPORTED;
  }
}

}  // namespace

kda_status launch_chunk_ffma(const void *q, const void *k, const void *v, const float *beta,
                             const float *log_alpha, const float *h0, void *o, float *hT,
                             int B, int H, int T, int dk, int dv, int C, kda_dtype dt,
                             kda_alpha_mode am, WorkspaceHeader * /*hdr*/,
                             cudaStream_t stream, LaunchTimer &timer) {
  const long long BH = (long long)B * H;
  if (chunk_ffma_launches((int)BH, T, hT != nullptr) == 0) return KDA_OK;
  if (BH > 65535) return KDA_ERR_UNSUPPORTED;  // grid.y limit
  if (dt == KDA_BF16)
    return launch_ffma_dt<__nv_bfloat16>(q, k, v, beta, log_alpha, h0, o, hT, (int)BH, T, dk,
                                         dv, C, am, stream, timer);
  return launch_ffma_dt<float>(q, k, v, beta, log_alpha, h0, o, hT, (int)BH, T, dk, dv, C, am,
                               stream, timer);
}

int chunk_ffma_launches(int BH, int T, bool has_hT) {
  return (BH == 0 || (T == 0 && !has_hT)) ? 0 : 1;
}

const char *chunk_ffma_kernel_name(int i) { return i == 0 ? "chunk_ffma_kernel" : nullptr; }

}  // namespace kda
