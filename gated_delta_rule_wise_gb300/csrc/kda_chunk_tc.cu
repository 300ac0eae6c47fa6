// kda_chunk_tc.cu -- tensor-core (tcgen05) chunked prefill of the gated delta
// rule for bf16 inputs, C = 64, dk = dv = D in {64, 128}.
//
// Method.  Per chunk of C tokens, with g the running sum of log(a) =
// -exp(log_alpha) from the chunk start (per key channel), gamma = exp(g) and
// gamma_C its value at the chunk end, the chunked form of the recurrence is
//   A  = strict_lower(diag(beta) (K*gamma) (K/gamma)^T),   T = (I + A)^-1
//   W  = T diag(beta) (K*gamma),   U = T diag(beta) V
//   u  = U - W S;   o = (Q*gamma) S + M u;   S' = Diag(gamma_C) S + Kbar^T u
// with M = lower_incl((Q*gamma)(K/gamma)^T) and Kbar = K*gamma_C/gamma.  For no
// decay it is the chunked DeltaNet loop of "22,580: From GPT-2 to Kimi K3"
// (yichencityu.github.io), section 6.3 (forward substitution on the C x C unit
// lower-triangular matrix; W = T K_beta; U = T V_beta; u = U - W S;
// o = q S + tril(q k^T) u; S += k^T u); the decay factors are the cumulative
// products the gated form needs ("22580: From GPT-2 to Kimi3, Explained"
// (zharfai.com), "Gated DeltaNet adds controlled forgetting"), per key channel
// as in "22580: From GPT-2 to Kimi K3, Explained" (lukebest.github.io),
// "KDA (per-channel alpha)".
//
// Substituting u, the pass over chunks needs one product with the state:
//   S' = (Diag(gamma_C) + Ap) S + Kbar^T U,      Ap = -Kbar^T W   (D x D)
//   o  = Qp S + M U,                              Qp = Q*gamma - M W  (C x D)
// Everything except S is known per chunk before the pass starts, so
//  - kda_prep_kernel (persistent CTAs, fully parallel over (head, chunk))
//    computes the decay prefix, the decayed tiles, A and M (one tcgen05 MMA
//    group), T by a blocked inverse in shared memory, W and U, then the
//    chunk's record: for D = 128 Ap and Qp as swizzled operand tiles and the
//    additive terms B = Kbar^T U and O = M U already multiplied out; for
//    D = 64 Ap, Qp, Kbar^T, M and U^T tiles.  gamma_C closes each record.
//  - kda_scan_kernel (one CTA per (head, block of 32 or 64 value columns)) walks the
//    chunks in order with the records streamed in by bulk copies; per chunk
//    it writes a bf16 copy of S as the MMA operand, forms
//    S' = gamma_C S + B + Ap S (one group of tcgen05 MMAs) and, off the
//    serial path, o = Qp S + O.  One MMA round trip per chunk sits on the
//    serial path.
// The D = 128 kernels are described in detail above prep_d128 and scan_d128.
// A call may also run in segments of the sequence, each segment's prep beside
// the previous segment's scan (the pipelined call, above launch_d).
// A partial last chunk is padded with k = q = v = 0, beta = 0, a = 1, which
// adds nothing; padded rows of o are not stored.
#include <type_traits>

#include "kda_launch.cuh"
#include "kda_ptx.cuh"
#include "kda_umma.cuh"

namespace kda {
namespace {

constexpr int kC = 64;                 // chunk length on this path
constexpr uint32_t kWaitLimit = 1u << 24;  // polls before a wait gives up (~1 s)

// Per-chunk intermediate record in the workspace, one per (head, chunk).
template <int D>
struct Rec;
// D = 64: every operand the scan multiplies, as swizzled K-major bf16 tiles
// (Ap and Qp, and Kbar^T and M, are adjacent 64-row tiles: one 128-row
// operand each), then gamma_C.
template <>
struct Rec<64> {
  static constexpr uint32_t AP = 0;        // Ap     [64 rows][64]
  static constexpr uint32_t QP = 8192;     // Qp     [C rows][64]
  static constexpr uint32_t KBT = 16384;   // Kbar^T [64 rows][C]
  static constexpr uint32_t MM = 24576;    // M      [C rows][C]
  static constexpr uint32_t UT = 32768;    // U^T    [64 rows][C]
  static constexpr uint32_t GC = 40960;    // gamma_C [64] float
  static constexpr uint32_t BYTES = 41216;
  static constexpr uint32_t PRE = UT;      // Ap | Qp | Kbar^T | M
};
// D = 128: the two operands of the state products as swizzled K-major tiles,
// then the chunk's additive terms already multiplied out: B = Kbar^T U
// [128 keys][128 values] and O = M U [C tokens][128 values], bf16 stored as
// four 32-column blocks each (a scan CTA owns one block) of 64-byte rows whose
// four 16-byte chunks are rotated: chunk q of row r sits at position
// q ^ ((r >> 1) & 3) (rotated_chunk), so that eight threads reading eight
// consecutive rows hit distinct banks; then gamma_C.
template <>
struct Rec<128> {
  static constexpr uint32_t AP = 0;        // Ap    [128 rows][128]
  static constexpr uint32_t QP = 32768;    // Qp    [C rows][128]
  static constexpr uint32_t BI = 49152;    // B     [4][128][32] bf16
  static constexpr uint32_t OI = 81920;    // O     [4][C][32] bf16
  static constexpr uint32_t GC = 98304;    // gamma_C [128] float
  static constexpr uint32_t BYTES = 98816;
  static constexpr uint32_t PRE = BI;      // Ap | Qp
  static constexpr int BLK = 32;           // value columns per block of B and O
};

__host__ __device__ constexpr uint32_t align1k(uint32_t x) { return (x + 1023u) & ~1023u; }
// Byte offset of 16-byte chunk q of row r in a block of 64-byte rows (B, O).
__host__ __device__ constexpr uint32_t rotated_chunk(int r, int q) {
  return (uint32_t)r * 64u + ((uint32_t)(q ^ ((r >> 1) & 3)) << 4);
}
constexpr int kLD = kC + 4;  // row stride (floats) of the float A and T tiles of the solve

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t *>(&p);
}
__device__ __forceinline__ void st_bf16(uint8_t *base, uint32_t off, float x) {
  *reinterpret_cast<__nv_bfloat16 *>(base + off) = __float2bfloat16_rn(x);
}
// 8 consecutive K values of one row -> one 16-byte chunk.
__device__ __forceinline__ void st_chunk(uint8_t *tile, int row, int c8, int rows, const float *v) {
  uint4 u;
  u.x = pack_bf16x2(v[0], v[1]);
  u.y = pack_bf16x2(v[2], v[3]);
  u.z = pack_bf16x2(v[4], v[5]);
  u.w = pack_bf16x2(v[6], v[7]);
  *reinterpret_cast<uint4 *>(tile + umma::sw128_chunk(row, c8, rows)) = u;
}
__device__ __forceinline__ void ld_chunk(const uint8_t *tile, int row, int c8, int rows, float *v) {
  const uint4 u = *reinterpret_cast<const uint4 *>(tile + umma::sw128_chunk(row, c8, rows));
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __nv_bfloat162 p = *reinterpret_cast<const __nv_bfloat162 *>(&w[i]);
    v[2 * i] = __low2float(p);
    v[2 * i + 1] = __high2float(p);
  }
}

// ============================================================== prep kernel

// Shared memory of the D = 64 prep (one CTA per SM).
struct PrepSmem64 {
  static constexpr int D = 64;
  using R = Rec<64>;
  // the whole record is staged here and leaves with one bulk copy
  static constexpr uint32_t AP_S = 0, QP_S = R::QP, GC_S = R::GC;
  static constexpr uint32_t KBT_S = R::KBT, MM_S = R::MM, UT_S = R::UT;
  static constexpr uint32_t X1 = align1k(R::BYTES);         // [K_beta; Q*gamma] [128 rows][D]
  static constexpr uint32_t TT = X1 + 128 * D * 2;         // T bf16 [C rows][C]; solve scratch before
  static constexpr uint32_t TF = TT + kC * kC * 2;         // T float [C][kLD] during the solve
  static constexpr uint32_t WT = TF;                       // W^T [D rows][C] afterwards
  static constexpr uint32_t AS = align1k(TF + kC * kLD * 4);  // A float [C][kLD]
  static constexpr uint32_t X2 = AS + kC * kLD * 4;        // [K_beta^T; (beta V)^T] [2D rows][C]
  static constexpr uint32_t KH = X2 + 2 * D * kC * 2;      // K/gamma  [C rows][D]
  static constexpr uint32_t RAW = KH + kC * D * 2;         // q | k | v [C][D] bf16
  static constexpr uint32_t BETA = RAW + 3 * kC * D * 2;   // float [C]
  static constexpr uint32_t PART = BETA + kC * 4;          // float [4][D] partial decay sums
  static constexpr uint32_t BAR = PART + 4 * D * 4;        // mbarrier (MMA commits)
  static constexpr uint32_t LBAR = BAR + 8;                // mbarrier (raw loads)
  static constexpr uint32_t TMEMP = LBAR + 8;              // TMEM base address
  static constexpr uint32_t BYTES = TMEMP + 8;
  static constexpr uint32_t TMEM_COLS = 128;
  static_assert(kC * kLD * 4 >= D * kC * 2, "W^T must fit the float T region");
  static_assert((X2 & 1023u) == 0 && (KH & 1023u) == 0 && (AS & 1023u) == 0 && (TF & 1023u) == 0 &&
                    (KBT_S & 1023u) == 0 && (MM_S & 1023u) == 0 && (UT_S & 1023u) == 0,
                "operand tiles need 1024-byte alignment");
  static_assert(BYTES + 1024 <= 232448, "prep shared memory");
};

__device__ __forceinline__ void fma4(float4 &acc, float a, const float4 &b) {
  acc.x += a * b.x; acc.y += a * b.y; acc.z += a * b.z; acc.w += a * b.w;
}

// T = (I + A)^-1 for the strictly lower A (float, row stride kLD), in blocks
// of 16: T_ij = -T_ii sum_{m=j..i-1} A_im T_mj.  The diagonal blocks T_ii and
// the six G_im = T_ii A_im below the diagonal, all at once by forward
// substitution (one right-hand column per thread, partial sums in registers);
// then T_ij = -sum_m G_im T_mj along the block subdiagonals (three blocks,
// then two, then one), every block product done by 64 threads on 1 x 4 strips.
// The float row stride kLD = C + 4 keeps column reads across rows and 16-byte
// row accesses free of bank conflicts, and lets every inner-loop address be an
// immediate offset.  Leaves T (float, lower blocks) in TF and the bf16 K-major
// [C][C] tile of T (zeros above the diagonal) in TT.  All 256 threads call
// it; G (6 blocks, rows kGLD floats apart) is scratch inside TT.
// `late` runs on threads 64..255 while threads 0..63 form the last block of
// T, after the last read of AF: the caller may reuse AF's space there.
struct NoLateWork {
  __device__ void operator()() const {}
};
constexpr int kGLD = 20;  // row stride (floats) of the G blocks: row reads conflict-free
static_assert(6 * 16 * kGLD * 4 <= kC * kC * 2, "G scratch fits the T tile");
template <class Late = NoLateWork>
__device__ __forceinline__ void blocked_unit_lower_inverse(const float *AF, float *TF, uint8_t *TT,
                                                           int tid, const Late &late = Late()) {
  float *XS = reinterpret_cast<float *>(TT);
  // One stage of 160 column solves, (I + A_ii) x = rhs by forward substitution
  // (partial sums in registers): 4 x 16 columns of the identity give the
  // diagonal blocks T_ii, 6 x 16 columns of A_im give G_im = T_ii A_im,
  // slots 0..5 = (1,0) (2,1) (3,2) (2,0) (3,1) (3,0).
  if (tid < 10 * 16) {
    const int blk = tid >> 4, j = tid & 15;
    const bool diag = blk < 4;
    const int sl = blk - 4;
    const int bi = diag ? blk : (sl < 3 ? sl + 1 : (sl == 5 ? 3 : sl - 1));
    const int bj = diag ? blk : (sl < 3 ? sl : (sl == 5 ? 0 : sl - 3));
    const float *Ab = AF + (bi * 16) * kLD + bi * 16;
    const float *rc = AF + (bi * 16) * kLD + bj * 16 + j;  // column j of A_(bi,bj)
    float t[16], p[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) p[i] = diag ? 0.f : -rc[i * kLD];
#pragma unroll
    for (int kk = 0; kk < 16; ++kk) {
      t[kk] = diag ? ((kk == j) ? 1.f : ((kk < j) ? 0.f : -p[kk])) : -p[kk];
#pragma unroll
      for (int i = kk + 1; i < 16; ++i) p[i] += Ab[i * kLD + kk] * t[kk];
    }
    if (diag) {
      float *Tb = TF + (bi * 16) * kLD + bi * 16 + j;
#pragma unroll
      for (int i = 0; i < 16; ++i) Tb[i * kLD] = t[i];
    } else {
      float *Gb = XS + sl * 16 * kGLD + j;
#pragma unroll
      for (int i = 0; i < 16; ++i) Gb[i * kGLD] = t[i];
    }
  }
  __syncthreads();
  const int r = (tid & 63) >> 2, c0 = (tid & 3) * 4, g = tid >> 6;
  // acc += sum_s L[r][s] R[s][c0..c0+3] over one 16 x 16 block pair
  auto strip = [&](float4 &acc, const float *lrow, const float *rblk) {
#pragma unroll
    for (int s2 = 0; s2 < 16; ++s2)
      fma4(acc, lrow[s2], *reinterpret_cast<const float4 *>(rblk + s2 * kLD + c0));
  };
  auto gs = [&](int slot) { return XS + slot * 16 * kGLD + r * kGLD; };  // row r of G slot
  auto tb = [&](int bi, int bj) { return TF + (bi * 16) * kLD + bj * 16; };  // block (bi, bj)
  auto put = [&](int bi, int bj, const float4 &acc) {
    *reinterpret_cast<float4 *>(TF + (bi * 16 + r) * kLD + bj * 16 + c0) =
        make_float4(-acc.x, -acc.y, -acc.z, -acc.w);
  };
  if (g < 3) {                                   // T_10, T_21, T_32 = -G_(i+1)i T_ii
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    strip(acc, gs(g), tb(g, g));
    put(g + 1, g, acc);
  }
  __syncthreads();
  if (g < 2) {                                   // T_20, T_31 = -(G_(i+2)i T_ii + G_(i+2)(i+1) T_(i+1)i)
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    strip(acc, gs(3 + g), tb(g, g));
    strip(acc, gs(1 + g), tb(g + 1, g));
    put(g + 2, g, acc);
  }
  __syncthreads();
  if (g == 0) {                                  // T_30 = -(G_30 T_00 + G_31 T_10 + G_32 T_20)
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    strip(acc, gs(5), tb(0, 0));
    strip(acc, gs(4), tb(1, 0));
    strip(acc, gs(2), tb(2, 0));
    put(3, 0, acc);
  } else {
    late();
  }
  __syncthreads();
  for (int u = tid; u < kC * 8; u += 256) {  // bf16 operand tile, zeros above the diagonal blocks
    const int row = u >> 3, c8 = u & 7;
    float x[8];
    if ((row >> 4) >= (c8 >> 1)) {
      const float4 a = *reinterpret_cast<const float4 *>(TF + row * kLD + c8 * 8);
      const float4 b = *reinterpret_cast<const float4 *>(TF + row * kLD + c8 * 8 + 4);
      x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
      x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
    } else {
#pragma unroll
      for (int e2 = 0; e2 < 8; ++e2) x[e2] = 0.f;
    }
    st_chunk(TT, row, c8, kC, x);
  }
}

// D = 64 prep: one CTA per SM, chunks taken in turn; the whole record is
// staged in shared memory and leaves with one bulk copy.
__device__ __forceinline__ void prep_d64(const __nv_bfloat16 *__restrict__ q,
                                         const __nv_bfloat16 *__restrict__ k,
                                         const __nv_bfloat16 *__restrict__ v,
                                         const float *__restrict__ beta,
                                         const float *__restrict__ log_alpha, int alpha_mode, int T,
                                         int NC, int total, uint8_t *__restrict__ ws, uint8_t *sm) {
  constexpr int D = 64;
  using Rr = Rec<D>;
  using L = PrepSmem64;
  constexpr int Q4 = 256 / D;          // threads per key channel
  constexpr int R = kC / Q4;           // rows per thread in the elementwise phase
  uint8_t *stg = sm;  // staging of the stored record
  uint8_t *X1 = sm + L::X1;
  uint8_t *TT = sm + L::TT;
  uint8_t *WT = sm + L::WT;
  float *AS = reinterpret_cast<float *>(sm + L::AS);
  float *TF = reinterpret_cast<float *>(sm + L::TF);
  uint8_t *X2 = sm + L::X2;
  uint8_t *KH = sm + L::KH;
  uint8_t *rawq = sm + L::RAW, *rawk = rawq + kC * D * 2, *rawv = rawk + kC * D * 2;
  float *part = reinterpret_cast<float *>(sm + L::PART);
  uint64_t *bar = reinterpret_cast<uint64_t *>(sm + L::BAR);
  uint64_t *lbar = reinterpret_cast<uint64_t *>(sm + L::LBAR);
  uint32_t *tmem_ptr = reinterpret_cast<uint32_t *>(sm + L::TMEMP);
  WorkspaceHeader *hdr = reinterpret_cast<WorkspaceHeader *>(ws);

  const int tid = threadIdx.x, warp = tid >> 5;
  const int c = tid % D, qtr = tid / D, r0 = qtr * R;
  // every thread waits on the same barriers; the chunk's last barrier ORs
  // the outcome of its waits so that the CTA leaves together after one gave up
  bool ok = true;
  auto fail = [&](unsigned where) {
    ok = false;
    report_error(hdr, KDA_ERR_TIMEOUT, where);
  };

  auto issue_raw = [&](int idx) {  // bulk copies of one chunk's q, k, v rows
    const int bh = idx / NC, t0 = (idx % NC) * kC;
    const int valid = min(kC, T - t0);
    const size_t row0 = (size_t)bh * T + t0;
    const uint32_t bytes = (uint32_t)valid * D * 2;
    ptx::mbar_arrive_expect_tx(lbar, 3 * bytes);
    ptx::bulk_g2s(rawq, q + row0 * D, bytes, lbar);
    ptx::bulk_g2s(rawk, k + row0 * D, bytes, lbar);
    ptx::bulk_g2s(rawv, v + row0 * D, bytes, lbar);
  };

  if (tid == 0) {
    ptx::mbar_init(bar, 1);
    ptx::mbar_init(lbar, 1);
    ptx::fence_mbar_init();
  }
  if (warp == 0) {
    ptx::tmem_alloc(tmem_ptr, L::TMEM_COLS);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_ptr;
  const uint32_t sX1 = ptx::smem_u32(X1), sKH = ptx::smem_u32(KH), sX2 = ptx::smem_u32(X2);
  const uint32_t sTT = ptx::smem_u32(TT), sWT = ptx::smem_u32(WT);
  const uint32_t sKBT = ptx::smem_u32(sm + L::KBT_S);
  if (tid == 0 && (int)blockIdx.x < total) issue_raw(blockIdx.x);
  uint32_t mma_phase = 0;

  // Decay inputs of the next chunk, prefetched in three batches hidden under the
  // three MMA waits of the current chunk (few loads in flight at a time):
  // log_alpha for this thread's key channel and rows, beta of row `tid`.
  float la_n[R], b_n = 0.f;
  auto load_la = [&](int idxn, auto I0, auto I1) {
    constexpr int i0 = decltype(I0)::value, i1 = decltype(I1)::value;
    const int t0n = (idxn % NC) * kC;
    const int validn = min(kC, T - t0n);
    const size_t row0n = (size_t)(idxn / NC) * T + t0n;
#pragma unroll
    for (int i = i0; i < i1; ++i) {
      const int rr = min(r0 + i, validn - 1);
      la_n[i] = 0.f;
      if (alpha_mode == KDA_ALPHA_CHANNEL)
        la_n[i] = log_alpha[(row0n + rr) * D + c];
      else if (alpha_mode == KDA_ALPHA_SCALAR)
        la_n[i] = log_alpha[row0n + rr];
    }
    if (i0 == 0 && tid < kC) b_n = beta[row0n + min(tid, validn - 1)];
  };
  using I_0 = std::integral_constant<int, 0>;
  using I_1 = std::integral_constant<int, R / 3>;
  using I_2 = std::integral_constant<int, 2 * R / 3>;
  using I_3 = std::integral_constant<int, R>;
  if ((int)blockIdx.x < total) load_la(blockIdx.x, I_0{}, I_3{});
  float *betas = reinterpret_cast<float *>(sm + L::BETA);

  for (int idx = blockIdx.x, it = 0; idx < total; idx += gridDim.x, ++it) {
    const int n = idx % NC;
    const int t0 = n * kC;
    const int valid = min(kC, T - t0);

    // ---- (1) decay inputs (loaded during the previous chunk), then the raw rows
    float ld[R];
#pragma unroll
    for (int i = 0; i < R; ++i)
      ld[i] = (r0 + i < valid && alpha_mode != KDA_ALPHA_NONE) ? -__expf(la_n[i]) : 0.f;
    if (tid < kC) betas[tid] = (tid < valid) ? b_n : 0.f;
    float psum = 0.f;
#pragma unroll
    for (int i = 0; i < R; ++i) psum += ld[i];
    part[qtr * D + c] = psum;
    if (tid == 0) ptx::bulk_wait_read_all();  // the previous record has left shared memory
    if (ok && !ptx::mbar_wait(lbar, it & 1, kWaitLimit)) fail(0x100u);
    for (int idx2 = valid * D + tid; idx2 < kC * D; idx2 += 256) {  // zero the padded rows
      reinterpret_cast<__nv_bfloat16 *>(rawq)[idx2] = __float2bfloat16_rn(0.f);
      reinterpret_cast<__nv_bfloat16 *>(rawk)[idx2] = __float2bfloat16_rn(0.f);
      reinterpret_cast<__nv_bfloat16 *>(rawv)[idx2] = __float2bfloat16_rn(0.f);
    }
    __syncthreads();
    float g = 0.f, gC = 0.f;
#pragma unroll
    for (int j = 0; j < Q4; ++j) {
      const float p = part[j * D + c];
      gC += p;
      if (j < qtr) g += p;
    }
    const float egC = __expf(gC);
    {
      float kbT[8], kbarT[8], vbT[8];
#pragma unroll
      for (int i = 0; i < R; ++i) {
        const int r = r0 + i;
        const float kv = __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(rawk)[r * D + c]);
        const float qv = __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(rawq)[r * D + c]);
        const float vv = __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(rawv)[r * D + c]);
        g += ld[i];
        const float eg = __expf(g), eng = __expf(-g);
        const float bti = betas[r];
        const float kb = bti * kv * eg;
        st_bf16(X1, umma::sw128_off(r, c, 128), kb);               // K_beta
        st_bf16(X1, umma::sw128_off(kC + r, c, 128), qv * eg);     // Q * gamma
        st_bf16(KH, umma::sw128_off(r, c, kC), kv * eng);          // K / gamma
        kbT[i & 7] = kb;
        kbarT[i & 7] = kv * eng * egC;
        vbT[i & 7] = bti * vv;
        if ((i & 7) == 7) {
          const int c8 = (r0 + i) >> 3;
          st_chunk(X2, c, c8, 2 * D, kbT);                          // K_beta^T
          st_chunk(X2, D + c, c8, 2 * D, vbT);                      // (beta V)^T
          st_chunk(sm + L::KBT_S, c, c8, D, kbarT);                 // Kbar^T (output)
        }
      }
      if (qtr == 0) reinterpret_cast<float *>(stg + L::GC_S)[c] = egC;
    }
    ptx::fence_proxy_async_smem();
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const int idx_next = idx + (int)gridDim.x;
    const bool has_next = idx_next < total;
    if (has_next && tid == 0) issue_raw(idx_next);  // prefetch the next chunk's q, k, v rows

    // ---- (2) [A_full; M_full] = [K_beta; Q*gamma] (K/gamma)^T  -> TMEM cols [0, 64)
    if (tid == 0) {
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks)
        ptx::mma_bf16_ss(tmem, umma::sdesc_k(sX1, 128, ks), umma::sdesc_k(sKH, kC, ks),
                         umma::idesc_bf16(128, kC), ks > 0);
      ptx::mma_commit(bar);
    }
    if (has_next) load_la(idx_next, I_0{}, I_1{});
    if (ok && !ptx::mbar_wait(bar, mma_phase & 1, kWaitLimit)) fail(0x101u);
    ++mma_phase;
    ptx::tc_fence_after();

    // ---- (3) rows 0..63: A (strict lower) as float; rows 64..127: M (and [I | -M])
    if (warp < 4) {
      const int lane_row = tid;
      const uint32_t ta = tmem + ((uint32_t)(warp * 32) << 16);
#pragma unroll
      for (int cb = 0; cb < kC; cb += 16) {
        float x[16];
        ptx::tmem_ld16(ta + cb, x);
        ptx::tmem_ld_wait();
        if (lane_row < kC) {
          const int r = lane_row;
#pragma unroll
          for (int j4 = 0; j4 < 4; ++j4) {
            const int m0 = cb + 4 * j4;
            float4 a;
            a.x = (m0 + 0 < r) ? x[4 * j4 + 0] : 0.f;
            a.y = (m0 + 1 < r) ? x[4 * j4 + 1] : 0.f;
            a.z = (m0 + 2 < r) ? x[4 * j4 + 2] : 0.f;
            a.w = (m0 + 3 < r) ? x[4 * j4 + 3] : 0.f;
            *reinterpret_cast<float4 *>(AS + r * kLD + m0) = a;
          }
        } else {
          const int r = lane_row - kC;
          float mrow[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) mrow[j] = (cb + j <= r) ? x[j] : 0.f;
          st_chunk(sm + L::MM_S, r, cb >> 3, kC, mrow);
          st_chunk(sm + L::MM_S, r, (cb >> 3) + 1, kC, mrow + 8);
        }
      }
    }
    __syncthreads();

    // ---- (4) T = (I + A)^-1 (blocked forward substitution)
    blocked_unit_lower_inverse(AS, TF, TT, tid);
    ptx::fence_proxy_async_smem();
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();

    // ---- (5) [W^T; U^T] = [K_beta^T; (beta V)^T] T^T  -> TMEM cols [64, 192) or [64, 128)
    if (tid == 0) {
#pragma unroll
      for (int h = 0; h < 2 * D / 128; ++h)
#pragma unroll
        for (int ks = 0; ks < kC / 16; ++ks)
          ptx::mma_bf16_ss(tmem + 64 + 64 * h, umma::sdesc_k(sX2 + h * 128 * 128, 2 * D, ks),
                           umma::sdesc_k(sTT, kC, ks), umma::idesc_bf16(128, kC), ks > 0);
      ptx::mma_commit(bar);
    }
    if (has_next) load_la(idx_next, I_1{}, I_2{});
    if (ok && !ptx::mbar_wait(bar, mma_phase & 1, kWaitLimit)) fail(0x102u);
    ++mma_phase;
    ptx::tc_fence_after();

    // ---- (6) W^T -> operand tile, U^T -> record
    if (warp < 4) {
      const uint32_t ta = tmem + ((uint32_t)(warp * 32) << 16);
#pragma unroll
      for (int h = 0; h < 2 * D / 128; ++h) {
#pragma unroll
        for (int cb = 0; cb < kC; cb += 16) {
          float x[16];
          ptx::tmem_ld16(ta + 64 + 64 * h + cb, x);
          ptx::tmem_ld_wait();
          // lanes 0..63 W^T rows, lanes 64..127 U^T rows
          const int lane_row = tid;
          const bool isW = lane_row < D;
          const int row = lane_row % D;
          uint8_t *dst = isW ? WT : sm + L::UT_S;
          st_chunk(dst, row, cb >> 3, D, x);
          st_chunk(dst, row, (cb >> 3) + 1, D, x + 8);
        }
      }
    }
    ptx::fence_proxy_async_smem();
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();

    // ---- (7) [Kbar^T; M] W
    if (tid == 0) {
      {
        // cols [0, 64): [Kbar^T; M] W  (Kbar^T and M are adjacent in the record)
#pragma unroll
        for (int ks = 0; ks < kC / 16; ++ks)
          ptx::mma_bf16_ss(tmem, umma::sdesc_k(sKBT, 128, ks), umma::sdesc_k(sWT, D, ks),
                           umma::idesc_bf16(128, D), ks > 0);
      }
      ptx::mma_commit(bar);
    }
    if (has_next) load_la(idx_next, I_2{}, I_3{});
    if (ok && !ptx::mbar_wait(bar, mma_phase & 1, kWaitLimit)) fail(0x103u);
    ++mma_phase;
    ptx::tc_fence_after();

    // ---- (8) Ap = -Kbar^T W;  Qp
    if (warp < 4) {
      const uint32_t ta = tmem + ((uint32_t)(warp * 32) << 16);
      const int lane_row = tid;
      {
#pragma unroll
        for (int cb = 0; cb < D; cb += 16) {
          float x[16];
          ptx::tmem_ld16(ta + cb, x);
          ptx::tmem_ld_wait();
          if (lane_row < D) {
#pragma unroll
            for (int j = 0; j < 16; ++j) x[j] = -x[j];
            st_chunk(stg + L::AP_S, lane_row, cb >> 3, D, x);
            st_chunk(stg + L::AP_S, lane_row, (cb >> 3) + 1, D, x + 8);
          } else {
            const int r = lane_row - D;
            float qg[16];
            ld_chunk(X1, kC + r, cb >> 3, 128, qg);
            ld_chunk(X1, kC + r, (cb >> 3) + 1, 128, qg + 8);
#pragma unroll
            for (int j = 0; j < 16; ++j) qg[j] -= x[j];
            st_chunk(stg + L::QP_S, r, cb >> 3, kC, qg);
            st_chunk(stg + L::QP_S, r, (cb >> 3) + 1, kC, qg + 8);
          }
        }
      }
    }
    ptx::fence_proxy_async_smem();
    ptx::tc_fence_before();
    const int stop = __syncthreads_or(!ok);  // a wait of this CTA gave up
    ptx::tc_fence_after();
    if (stop) {
      // drain (bounded) what thread 0 started: the latest row copy, the products
      if (tid == 0) {
        ptx::mbar_wait(lbar, (it + (has_next ? 1 : 0)) & 1, kWaitLimit);
        ptx::mma_commit(bar);
        ptx::mbar_wait(bar, mma_phase & 1, kWaitLimit);
      }
      break;
    }

    // ---- (9) record -> workspace (one bulk copy; its read is awaited before
    // the record region is written again)
    if (tid == 0) {
      uint8_t *dst = ws + sizeof(WorkspaceHeader) + (size_t)idx * Rr::BYTES;
      ptx::bulk_s2g(dst, stg, Rr::BYTES);
      ptx::bulk_commit();
    }
  }
  if (tid == 0) ptx::bulk_wait_all();
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, L::TMEM_COLS);
  }
}

// D = 128 prep.  Two CTAs share an SM (about 109 KB of shared memory, 256 TMEM
// columns and at most 128 registers per thread each), so one CTA's MMA waits,
// barriers and loads overlap the other's work.  Per chunk:
//  (0) decay, one thread per key channel and half of the rows: g = running sum
//      of -exp(log_alpha), gamma = exp(g) to a float tile over the
//      log_alpha rows; gamma_C to the record;
//  (1) the chunk's q, k, v rows to registers, then one thread per (row, 8
//      channels) writes K_beta = beta K gamma, Q*gamma, beta V and K/gamma as
//      natural (row = token) swizzled tiles over them;
//  (2) [A; M] = [K_beta; Q*gamma] (K/gamma)^T        8 MMAs (M = 128, N = 64)
//  (3) A to float;  (4) T = (I + A)^-1 (blocked), M to a bf16 tile in A's
//      space while the last block of T is formed
//  (5) [W | U] = T [K_beta | beta V]                   4 MMAs (M = 64, N = 256),
//      the right factor read MN-major from the natural tiles
//  (6) [W | U] to a natural tile over K_beta and beta V
//  (7) (K/gamma)^T [W | U]                              4 MMAs (M = 128, N = 256)
//  (8) Ap = -gamma_C (K/gamma)^T W and B = gamma_C (K/gamma)^T U to the record
//  (9) M [W | U]                                        4 MMAs (M = 64, N = 256)
// (10) Qp = Q*gamma - M W and O = M U to the record.
// Each warp assembles its contiguous pieces of the record tiles in staging
// slots of consumed shared memory, and bulk stores copy them out while the
// CTA goes on.
// The next chunk's input rows are prefetched into L2 during (5); its log_alpha,
// k and v rows are bulk-copied as soon as the last product has read A's space
// and blocks 2-3 (after (9)), its q rows after (10).
// Normalised linear attention: per (head, chunk) two vectors the scan needs
// besides the record, in a region that follows all records of the workspace:
// the row sums of the chunk's M (the intra-chunk part of each denominator) and
// sum_s Kbar_s (the chunk's contribution to the normaliser z).
struct NormRec {
  static constexpr uint32_t MR = 0;            // float [C]
  static constexpr uint32_t KS = kC * 4;       // float [128]
  static constexpr uint32_t BYTES = KS + 128 * 4;
};
static_assert(NormRec::BYTES % 16 == 0, "bulk-copied");

struct PrepSmem128 {
  using R = Rec<128>;
  static constexpr int D = 128;
  // X1: blocks 0-1 = [K_beta; Q*gamma] (128 rows x 128), blocks 2-3 = [beta V;
  // K/gamma]; rows 0-63 of the four blocks hold [W | U] (64 rows x 256) from
  // phase 6 on.  Before phase 1 blocks 0, 2 and 3 receive the raw q, k and v rows.
  static constexpr uint32_t X1 = 0;
  static constexpr uint32_t RAWQ = X1, RAWK = X1 + 32768, RAWV = X1 + 49152;
  // R_A: log_alpha as float [C][D], then gamma in two channel planes (channels
  // 8k..8k+3 | 8k+4..8k+7 of each row; the second plane 64 B further, so the
  // per-channel writes and the 16-byte row reads are both conflict-free)
  // (phases 0-1) | A, T float (3-4) | M tile (4-9)
  static constexpr uint32_t RA = X1 + 65536;
  static constexpr uint32_t EG = RA, AF = RA, TF = RA + kC * kLD * 4, MM = RA;
  static constexpr uint32_t EG_PLANE = kC * (D / 2) * 4 + 64;  // bytes from plane 0 to plane 1
  static constexpr uint32_t TT = align1k(RA + 2 * kC * kLD * 4);  // T bf16; solve scratch before
  static constexpr uint32_t GCS = TT + kC * kC * 2;  // gamma_C / gamma_mid float [D]
  static constexpr uint32_t GMID = GCS + D * 4;      // gamma_mid float [D]
  static constexpr uint32_t BETA = GMID + D * 4;     // float [C]
  static constexpr uint32_t PART = BETA + kC * 4;    // float [2][D]
  static constexpr uint32_t BAR = PART + 2 * D * 4;
  static constexpr uint32_t LBAR = BAR + 8;   // log_alpha, k, v rows landed
  static constexpr uint32_t QBAR = LBAR + 8;  // q rows landed
  static constexpr uint32_t TMEMP = QBAR + 8;
  static constexpr uint32_t NEXT = TMEMP + 4;  // the CTA's next work item
  static constexpr uint32_t BYTES = TMEMP + 8;
  static constexpr uint32_t TMEM_COLS = 256;
  static_assert(kC * D * 4 <= 2 * kC * kLD * 4 && EG_PLANE + kC * (D / 2) * 4 <= 2 * kC * kLD * 4,
                "log_alpha and gamma tiles fit R_A");
  static_assert(kC * kC * 2 <= kC * kLD * 4, "M tile fits A's space");
  static_assert((RA & 1023u) == 0 && (TT & 1023u) == 0, "tile alignment");
  // two CTAs per SM: 228 KB per SM, 1 KB reserved per CTA, 1 KB alignment slack
  static_assert(2 * (BYTES + 1024 + 1024) <= 233472, "prep shared memory");
};

__device__ __forceinline__ void unpack8(const uint4 &u, float *f) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __nv_bfloat162 p = *reinterpret_cast<const __nv_bfloat162 *>(&w[i]);
    f[2 * i] = __low2float(p);
    f[2 * i + 1] = __high2float(p);
  }
}
// silu(x) = x sigmoid(x) = h + h tanh(h), h = x / 2: one tanh.approx (relative
// error about 2^-11, below the bf16 rounding the tiles go through) in place of
// an exponential and a reciprocal.
__device__ __forceinline__ float silu_tanh(float x) {
  const float h = 0.5f * x;
  float t;
  asm("tanh.approx.f32 %0, %1;" : "=f"(t) : "f"(h));
  return fmaf(h, t, h);
}
__device__ __forceinline__ uint4 pack8(const float *x) {
  return make_uint4(pack_bf16x2(x[0], x[1]), pack_bf16x2(x[2], x[3]), pack_bf16x2(x[4], x[5]),
                    pack_bf16x2(x[6], x[7]));
}

// kMode 0 compiles the plain gated delta rule (rule and maps fixed at 0, their
// code folded away); 1 the delta rule with the silu / sigmoid maps read at run
// time (the linear rules' code folded away); 2 the linear rules (no solve
// compiled in) with the silu and ELU + 1 maps and the normalised rule's sums.  The modes are separate instantiations
// because the prep runs at the register limit: code that only one mode needs
// would cost the others spills.  kRowDecay: scalar or no decay (one factor per
// token row) rather than one per key channel; a separate instantiation too
// (both decay paths in one kernel made the per-channel one 4 % slower).
template <int kMode, bool kRowDecay>
__device__ __forceinline__ void prep_d128(const __nv_bfloat16 *__restrict__ q,
                                          const __nv_bfloat16 *__restrict__ k,
                                          const __nv_bfloat16 *__restrict__ v,
                                          const float *__restrict__ beta,
                                          const float *__restrict__ log_alpha, int alpha_mode,
                                          int T, int NC, int total, int n0, int nseg, int work,
                                          unsigned *ctr, uint8_t *__restrict__ ws, uint8_t *sm,
                                          int rule, unsigned maps) {
  constexpr int D = 128;
  constexpr bool kGeneral = kMode != 0, kExt = kMode == 2;
  using Rr = Rec<128>;
  using L = PrepSmem128;
  constexpr int R = 32;                // rows per thread in the decay phase
  float *EG = reinterpret_cast<float *>(sm + L::EG);
  float *AF = reinterpret_cast<float *>(sm + L::AF);
  float *TF = reinterpret_cast<float *>(sm + L::TF);
  uint8_t *TT = sm + L::TT, *MM = sm + L::MM, *X1 = sm + L::X1;
  const uint8_t *rawq = sm + L::RAWQ, *rawk = sm + L::RAWK, *rawv = sm + L::RAWV;
  float *gcs = reinterpret_cast<float *>(sm + L::GCS);
  float *gmid = reinterpret_cast<float *>(sm + L::GMID);
  float *betas = reinterpret_cast<float *>(sm + L::BETA);
  float *part = reinterpret_cast<float *>(sm + L::PART);
  uint64_t *bar = reinterpret_cast<uint64_t *>(sm + L::BAR);
  uint64_t *lbar = reinterpret_cast<uint64_t *>(sm + L::LBAR);
  uint64_t *qbar = reinterpret_cast<uint64_t *>(sm + L::QBAR);
  uint32_t *tmem_ptr = reinterpret_cast<uint32_t *>(sm + L::TMEMP);
  int *next_s = reinterpret_cast<int *>(sm + L::NEXT);
  WorkspaceHeader *hdr = reinterpret_cast<WorkspaceHeader *>(ws);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int quarter = warp & 3, colhalf = warp >> 2;  // TMEM lane quarter, column half
  const int c = tid & (D - 1), half = tid >> 7, r0 = half * R;   // decay phase mapping
  // Every thread waits on the same barriers, so a wait that gives up gives
  // up in every thread; the chunk's last barrier ORs the outcome and the
  // whole CTA leaves together (after draining what thread 0 started).
  bool ok = true;
  auto fail = [&](unsigned where) {
    ok = false;
    report_error(hdr, KDA_ERR_TIMEOUT, where);
  };

  constexpr bool la_bulk = !kRowDecay;  // per-channel log_alpha rows (512 B each), bulk-copied
  // The grid's work items are chunks n0 .. n0 + nseg - 1 of every head (all
  // chunks when n0 = 0 and nseg = NC); item l is record (head, chunk) of index
  auto chunk_of = [&](int l) { return (l / nseg) * NC + n0 + l % nseg; };
  auto rows_of = [&](int idx, int &valid, size_t &row0) {
    const int t0 = (idx % NC) * kC;
    valid = min(kC, T - t0);
    row0 = (size_t)(idx / NC) * T + t0;
  };
  auto issue_lkv = [&](int idx) {  // log_alpha -> R_A, k -> block 2, v -> block 3
    int valid;
    size_t row0;
    rows_of(idx, valid, row0);
    const uint32_t bytes = (uint32_t)valid * D * 2;
    ptx::mbar_arrive_expect_tx(lbar, 2 * bytes + (la_bulk ? 2 * bytes : 0u));
    if (la_bulk) ptx::bulk_g2s(sm + L::EG, log_alpha + row0 * D, 2 * bytes, lbar);
    ptx::bulk_g2s(sm + L::RAWK, k + row0 * D, bytes, lbar);
    ptx::bulk_g2s(sm + L::RAWV, v + row0 * D, bytes, lbar);
  };
  auto issue_q = [&](int idx) {  // q -> block 0
    int valid;
    size_t row0;
    rows_of(idx, valid, row0);
    const uint32_t bytes = (uint32_t)valid * D * 2;
    ptx::mbar_arrive_expect_tx(qbar, bytes);
    ptx::bulk_g2s(sm + L::RAWQ, q + row0 * D, bytes, qbar);
  };
  auto prefetch_rows = [&](int idx) {  // a chunk's input rows into L2 ahead of its copies
    int valid;
    size_t row0;
    rows_of(idx, valid, row0);
    const uint32_t bytes = (uint32_t)valid * D * 2;
    if (la_bulk) ptx::prefetch_l2(log_alpha + row0 * D, 2 * bytes);
    ptx::prefetch_l2(k + row0 * D, bytes);
    ptx::prefetch_l2(v + row0 * D, bytes);
    ptx::prefetch_l2(q + row0 * D, bytes);
  };

  if (tid == 0) {
    ptx::mbar_init(bar, 1);
    ptx::mbar_init(lbar, 1);
    ptx::mbar_init(qbar, 1);
    ptx::fence_mbar_init();
  }
  if (warp == 0) {
    ptx::tmem_alloc(tmem_ptr, L::TMEM_COLS);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_ptr;
  const uint32_t t_lane = tmem + ((uint32_t)(quarter * 32) << 16);
  const uint32_t sX1 = ptx::smem_u32(X1), sTT = ptx::smem_u32(TT), sMM = ptx::smem_u32(MM);
  const uint32_t sWU = sX1;                          // [W | U]: rows 0-63 of the four blocks
  const uint32_t sKH = sX1 + 32768 + kC * 128;       // K/gamma: rows 64-127 of blocks 2-3
  if (tid == 0 && (int)blockIdx.x < work) {
    issue_lkv(chunk_of(blockIdx.x));
    issue_q(chunk_of(blockIdx.x));
  }
  if constexpr (!kGeneral) {
    rule = KDA_RULE_DELTA;
    maps = 0u;
  }
  if constexpr (kMode == 1) rule = KDA_RULE_DELTA;
  const bool linear = kExt || rule != KDA_RULE_DELTA;  // W = 0, U = V: no beta, no solve
  const bool norm = kExt && rule == KDA_RULE_LINEAR_NORM;  // also the normaliser's sums
  uint8_t *const nrm0 = ws + sizeof(WorkspaceHeader) + (size_t)total * Rr::BYTES;
  auto beta_of = [&](int idx) -> float {        // beta of row tid of a chunk (tid < C)
    int vn;
    size_t rn;
    rows_of(idx, vn, rn);
    if (tid >= vn) return 0.f;
    if (linear) return 1.f;
    const float b = beta[rn + tid];
    return (maps & KDA_MAP_BETA_SIGMOID) ? 1.f / (1.f + __expf(-b)) : b;
  };
  float b_next = 0.f;  // beta of the next chunk's row tid (tid < C)
  // scalar decay: log_alpha of the next chunk's row tid, loaded with its beta
  // (not bulk-copied; read at the start of the decay phase it sat on the path)
  auto la_row_of = [&](int idx) -> float {
    int vn;
    size_t rn;
    rows_of(idx, vn, rn);
    return (alpha_mode == KDA_ALPHA_SCALAR && tid < vn) ? log_alpha[rn + tid] : 0.f;
  };
  float la_next = 0.f;
  if ((int)blockIdx.x < work && tid < kC) {
    b_next = beta_of(chunk_of(blockIdx.x));
    if constexpr (kRowDecay) la_next = la_row_of(chunk_of(blockIdx.x));
  }
  uint32_t mma_phase = 0;

  auto wait_mma = [&](unsigned code) {
    if (ok && !ptx::mbar_wait(bar, mma_phase & 1, kWaitLimit)) fail(code);
    ++mma_phase;
    ptx::tc_fence_after();
  };
  auto sync_for_mma = [&]() {  // generic smem writes -> async proxy; TMEM ops ordered
    ptx::fence_proxy_async_smem();
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
  };

  // Work items: the CTA's first is its index; each later one is claimed from
  // a counter (zero at the call's start), so that the two CTAs of an SM,
  // which do not run at the same speed (the older one's warps win the issue
  // slots), finish within a chunk of each other.  The claim for the next
  // item goes out at the top of a chunk and is read after the decay phase.
  int l = blockIdx.x;
  for (int it = 0; l < work; ++it) {
    int claimed = 0;
    if (tid == 0) claimed = (int)gridDim.x + (int)atomicAdd(ctr, 1u);
    const int idx = chunk_of(l);
    const int n = idx % NC;
    const int t0 = n * kC;
    const int valid = min(kC, T - t0);
    const size_t row0 = (size_t)(idx / NC) * T + t0;
    uint8_t *recg = ws + sizeof(WorkspaceHeader) + (size_t)idx * Rr::BYTES;


    // ---- (0) decay
    if (tid < kC) betas[tid] = b_next;
    if (ok && !ptx::mbar_wait(lbar, it & 1, kWaitLimit)) fail(0x100u);
    // gamma is measured from the middle of the chunk (g at row C/2 - 1 = p0):
    // the split factors gamma and 1/gamma then stay within exp(|half-chunk
    // decay|), so float and bf16 hold them up to a decay of about 87 per half
    // chunk; the chunk-start values are restored where they are needed
    if (la_bulk) {  // one decay per key channel: a prefix per channel
      float ld[R];
#pragma unroll
      for (int i = 0; i < R; ++i) ld[i] = EG[(r0 + i) * D + c];  // one straight run of shared loads
      float psum = 0.f;
#pragma unroll
      for (int i = 0; i < R; ++i) {
        ld[i] = (r0 + i < valid) ? -__expf(ld[i]) : 0.f;
        psum += ld[i];
      }
      part[half * D + c] = psum;
      __syncthreads();
      const float p0 = part[c], p1 = part[D + c];
      float g = half ? 0.f : -p0;
#pragma unroll
      for (int i = 0; i < R; ++i) {
        g += ld[i];
        EG[((c >> 2) & 1) * (L::EG_PLANE / 4) + (r0 + i) * (D / 2) + (c >> 3) * 4 + (c & 3)] =
            __expf(g);
      }
      if (half == 0) {
        gcs[c] = __expf(p1);   // gamma_C / gamma_mid: scales (K/gamma)^T into Kbar^T
        gmid[c] = __expf(p0);  // gamma_mid: turns Q*gamma (mid-referenced) into Q*gamma
        reinterpret_cast<float *>(recg + Rr::GC)[c] = __expf(p0 + p1);
      }
    } else {
      // one decay per token (scalar mode) or none: the prefix over the chunk's
      // rows runs once, one thread per row in the first two warps (a warp scan
      // each, the first warp's total carried into the second), and the tiles
      // take gamma and 1/gamma per row from EG[r] and EG[C + r]
      float x = 0.f;
      if (tid < kC) {
        if (alpha_mode == KDA_ALPHA_SCALAR && tid < valid) x = -__expf(la_next);
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          const float y = __shfl_up_sync(0xffffffffu, x, off);
          if (lane >= off) x += y;
        }
        if (lane == 31) part[warp] = x;  // rows 0-31 (= g at row C/2 - 1) and rows 32-63
      }
      __syncthreads();
      const float p0 = part[0], p1 = part[1];
      if (tid < kC) {
        const float g = warp == 0 ? x - p0 : x;  // g_r - g_mid
        EG[tid] = __expf(g);
        EG[kC + tid] = __expf(-g);
      }
      if (tid < D) {
        gcs[tid] = __expf(p1);
        gmid[tid] = __expf(p0);
        reinterpret_cast<float *>(recg + Rr::GC)[tid] = __expf(p0 + p1);
      }
    }
    if (tid == 0) *next_s = claimed;
    if (ok && !ptx::mbar_wait(qbar, it & 1, kWaitLimit)) fail(0x105u);
    __syncthreads();
    const int l_next = *next_s;
    const bool has_next = l_next < work;
    const int idx_next = has_next ? chunk_of(l_next) : 0;

    // ---- (1) decayed tiles, one thread per (row, 8 channels): raw rows to
    // registers first (the tiles overwrite them), rows past the end as zeros
    uint4 rq[4], rk[4], rv[4];
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const int u = tid + 256 * m;
      const int r = u >> 4, c8 = u & 15;
      const uint32_t off = (uint32_t)r * (D * 2) + (uint32_t)c8 * 16u;
      const bool in = r < valid;
      rq[m] = in ? *reinterpret_cast<const uint4 *>(rawq + off) : make_uint4(0u, 0u, 0u, 0u);
      rk[m] = in ? *reinterpret_cast<const uint4 *>(rawk + off) : make_uint4(0u, 0u, 0u, 0u);
      rv[m] = in ? *reinterpret_cast<const uint4 *>(rawv + off) : make_uint4(0u, 0u, 0u, 0u);
    }
    // the previous chunk's Qp and O stores have read their slots in block 1
    // and the T tile before the tiles below overwrite block 1
    if (lane == 0) ptx::bulk_wait_read<0>();
    __syncthreads();
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const int u = tid + 256 * m;
      const int r = u >> 4, c8 = u & 15;
      float kf[8], qf[8], vf[8], eg[8];
      unpack8(rk[m], kf);
      unpack8(rq[m], qf);
      unpack8(rv[m], vf);
      if (kExt && (maps & KDA_MAP_QK_ELU1)) {  // q, k <- elu(x) + 1 = max(x, 0) + exp(min(x, 0));
        const float in = r < valid ? 1.f : 0.f;  // rows past the end stay zero
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          qf[e] = in * (fmaxf(qf[e], 0.f) + __expf(fminf(qf[e], 0.f)));
          kf[e] = in * (fmaxf(kf[e], 0.f) + __expf(fminf(kf[e], 0.f)));
        }
      }
      if (maps & KDA_MAP_QK_SILU_NORM) {  // q, k <- silu / ||silu||, the row's 16 lanes reduce
        float sq = 0.f, sk = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          qf[e] = silu_tanh(qf[e]);
          kf[e] = silu_tanh(kf[e]);
          sq += qf[e] * qf[e];
          sk += kf[e] * kf[e];
        }
#pragma unroll
        for (int off = 1; off < 16; off <<= 1) {
          sq += __shfl_xor_sync(0xffffffffu, sq, off);
          sk += __shfl_xor_sync(0xffffffffu, sk, off);
        }
        const float iq = rsqrtf(fmaxf(sq, 1e-24f)), ik = rsqrtf(fmaxf(sk, 1e-24f));
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          qf[e] *= iq;
          kf[e] *= ik;
        }
      }
      float igr = 0.f;  // per-row 1 / gamma (scalar or no decay)
      if (la_bulk) {
        const float4 e0 = *reinterpret_cast<const float4 *>(EG + r * (D / 2) + c8 * 4);
        const float4 e1 =
            *reinterpret_cast<const float4 *>(EG + L::EG_PLANE / 4 + r * (D / 2) + c8 * 4);
        eg[0] = e0.x; eg[1] = e0.y; eg[2] = e0.z; eg[3] = e0.w;
        eg[4] = e1.x; eg[5] = e1.y; eg[6] = e1.z; eg[7] = e1.w;
      } else {  // per-row factors
        const float gr = EG[r];
        igr = EG[kC + r];
#pragma unroll
        for (int e = 0; e < 8; ++e) eg[e] = gr;
      }
      const float bt = betas[r];
      float kb[8], qg[8], vb[8], kh[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        // linear rules: W = 0, except that the normalised rule puts a ones
        // column (channel 0, valid rows) there: the products (K/gamma)^T W and
        // M W then leave the chunk's key sums and M's row sums in column 0
        kb[e] = linear ? ((norm && c8 == 0 && e == 0 && r < valid) ? 1.f : 0.f)
                       : bt * kf[e] * eg[e];
        qg[e] = qf[e] * eg[e];
        vb[e] = bt * vf[e];
        kh[e] = kf[e] * (la_bulk ? __fdividef(1.f, eg[e]) : igr);
      }
      st_chunk(X1, r, c8, 128, kb);                 // K_beta          (blocks 0-1, rows 0-63)
      st_chunk(X1, kC + r, c8, 128, qg);            // Q * gamma       (blocks 0-1, rows 64-127)
      st_chunk(X1 + 32768, r, c8, 128, vb);         // beta V          (blocks 2-3, rows 0-63)
      st_chunk(X1 + 32768, kC + r, c8, 128, kh);    // K / gamma       (blocks 2-3, rows 64-127)
    }
    sync_for_mma();

    // ---- (2) [A; M] = [K_beta; Q*gamma] (K/gamma)^T   -> TMEM cols [0, 64)
    if (tid == 0) {
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks)
        ptx::mma_bf16_ss(tmem, umma::sdesc_k(sX1, 128, ks), umma::sdesc_k(sKH, 128, ks),
                         umma::idesc_bf16(128, kC), ks > 0);
      ptx::mma_commit(bar);
    }
    wait_mma(0x101u);

    auto read_m = [&]() {  // lanes 64..127 (M, lower incl.) -> bf16 tile in A's space
      if (quarter >= 2) {
        const int r = quarter * 32 + lane - kC;
        const int cb = colhalf * 32;
        float x[32];
        ptx::tmem_ld32(t_lane + cb, x);
        ptx::tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 32; ++j) x[j] = (cb + j <= r) ? x[j] : 0.f;
#pragma unroll
        for (int j8 = 0; j8 < 4; ++j8) st_chunk(MM, r, (cb >> 3) + j8, kC, x + 8 * j8);
      }
    };
    if (linear) {  // [W | U] = [0 | V] already sits in rows 0-63 of the tile area
      read_m();
      sync_for_mma();
    } else {

    // ---- (3) lanes 0..63: A (strict lower) as float, 32 columns per warp
    if (quarter < 2) {
      const int r = quarter * 32 + lane;
      const int cb = colhalf * 32;
      float x[32];
      ptx::tmem_ld32(t_lane + cb, x);
      ptx::tmem_ld_wait();
#pragma unroll
      for (int j4 = 0; j4 < 8; ++j4) {
        const int m0 = cb + 4 * j4;
        float4 a;
        a.x = (m0 + 0 < r) ? x[4 * j4 + 0] : 0.f;
        a.y = (m0 + 1 < r) ? x[4 * j4 + 1] : 0.f;
        a.z = (m0 + 2 < r) ? x[4 * j4 + 2] : 0.f;
        a.w = (m0 + 3 < r) ? x[4 * j4 + 3] : 0.f;
        *reinterpret_cast<float4 *>(AF + r * kLD + m0) = a;
      }
    }
    __syncthreads();

    // ---- (4) T = (I + A)^-1; lanes 64..127 (M, lower incl.) to a bf16 tile
    // in A's space once A is no longer read
    blocked_unit_lower_inverse(AF, TF, TT, tid, read_m);
    sync_for_mma();

    // ---- (5) [W | U] = T [K_beta | beta V]   -> TMEM cols [0, 256), M = 64 layout
    if (tid == 0) {
#pragma unroll
      for (int ks = 0; ks < kC / 16; ++ks)
        ptx::mma_bf16_ss(tmem, umma::sdesc_k(sTT, kC, ks), umma::sdesc_mn(sX1, 128, ks),
                         umma::idesc_bf16_bmn(64, 256), ks > 0);
      ptx::mma_commit(bar);
    }
    if (tid == 32 && has_next) prefetch_rows(idx_next);
    wait_mma(0x102u);

    // ---- (6) [W | U] rows -> natural tile over K_beta and beta V (both consumed).
    // M = 64 layout: a warp's 16 rows sit in lanes 0-15 of its quarter; threads
    // 0-15 read columns c.., threads 16-31 the same rows at c + 64..
    {
      const int rr = quarter * 16 + (lane & 15), side = lane >> 4;
      float x[32], y[32];
      ptx::tmem_ld32_halves<64>(t_lane + colhalf * 128, x);
      ptx::tmem_ld32_halves<64>(t_lane + colhalf * 128 + 32, y);
      ptx::tmem_ld_wait();
      const int c8 = (colhalf * 128 + side * 64) >> 3;  // first chunk of this thread's 64 columns
      if (colhalf == 0) {  // W: K_beta carried gamma / gamma_mid; back to chunk-start gamma
        const float4 *gm = reinterpret_cast<const float4 *>(gmid + side * 64);
#pragma unroll
        for (int j4 = 0; j4 < 8; ++j4) {
          const float4 a = gm[j4], b = gm[8 + j4];
          x[4 * j4] *= a.x; x[4 * j4 + 1] *= a.y; x[4 * j4 + 2] *= a.z; x[4 * j4 + 3] *= a.w;
          y[4 * j4] *= b.x; y[4 * j4 + 1] *= b.y; y[4 * j4 + 2] *= b.z; y[4 * j4 + 3] *= b.w;
        }
      }
#pragma unroll
      for (int j8 = 0; j8 < 4; ++j8) st_chunk(X1, rr, c8 + j8, 128, x + 8 * j8);
#pragma unroll
      for (int j8 = 0; j8 < 4; ++j8) st_chunk(X1, rr, c8 + 4 + j8, 128, y + 8 * j8);
    }
    sync_for_mma();
    }  // delta rule

    // ---- (7) (K/gamma)^T [W | U] -> cols [0, 256)
    if (tid == 0) {
#pragma unroll
      for (int ks = 0; ks < kC / 16; ++ks)
        ptx::mma_bf16_ss(tmem, umma::sdesc_mn(sKH, 128, ks), umma::sdesc_mn(sWU, 128, ks),
                         umma::idesc_bf16_abmn(128, 256), ks > 0);
      ptx::mma_commit(bar);
    }
    wait_mma(0x103u);

    // ---- (8) lane = key channel: Ap = -gamma_C (K/gamma)^T W (warps 0-3),
    // B = gamma_C (K/gamma)^T U (warps 4-7).  A warp's rows form contiguous
    // pieces of the record (4 KB of Ap per K atom, 2 KB of B per 32-column
    // block): each piece is assembled in one of two staging slots of the warp
    // (shared memory no longer needed by this chunk: the consumed K/gamma rows,
    // the T tile, A's and T's float space past the M tile) and handed by lane 0
    // to a bulk store, so no warp waits for its global writes; a slot is
    // written again only after its earlier store has read it, and all stores
    // have read their slots before the next chunk's rows land there (after
    // (9)).  Copied out by the warps themselves, the 64 KB took about a
    // microsecond of this phase.
    {
      const int key = quarter * 32 + lane;
      const float gk = colhalf == 0 ? -gcs[key] : gcs[key];
      if (colhalf == 0) {
        uint8_t *slots = quarter < 2 ? X1 + 40960 + quarter * 16384 : sm + L::RA + 8192 * (quarter - 1);
#pragma unroll 1
        for (int a = 0; a < 2; ++a) {
          float x[64];
          ptx::tmem_ld32(t_lane + a * 64, *reinterpret_cast<float(*)[32]>(x));
          ptx::tmem_ld32(t_lane + a * 64 + 32, *reinterpret_cast<float(*)[32]>(x + 32));
          ptx::tmem_ld_wait();
          if (norm && a == 0) {  // sum_s Kbar_s = gamma_C/gamma_mid * sum_s (K/gamma)_s
            reinterpret_cast<float *>(nrm0 + (size_t)idx * NormRec::BYTES + NormRec::KS)[key] =
                gcs[key] * x[0];
            x[0] = 0.f;
          }
#pragma unroll
          for (int j = 0; j < 64; ++j) x[j] *= gk;
          uint8_t *stg = slots + a * 4096;
#pragma unroll
          for (int j8 = 0; j8 < 8; ++j8)  // same swizzle as the record tile (rows 32q + lane)
            *reinterpret_cast<uint4 *>(stg + lane * 128 + ((j8 ^ (lane & 7)) << 4)) = pack8(x + 8 * j8);
          ptx::fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            ptx::bulk_s2g(recg + Rr::AP + a * (D * 128) + quarter * 4096, stg, 4096);
            ptx::bulk_commit();
          }
        }
      } else {
        uint8_t *slots = quarter < 2 ? TT + quarter * 4096 : sm + L::RA + 24576 + (quarter - 2) * 4096;
#pragma unroll 1
        for (int h2 = 0; h2 < 2; ++h2) {
          float x[64];
          ptx::tmem_ld32(t_lane + 128 + h2 * 64, *reinterpret_cast<float(*)[32]>(x));
          ptx::tmem_ld32(t_lane + 128 + h2 * 64 + 32, *reinterpret_cast<float(*)[32]>(x + 32));
          ptx::tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 64; ++j) x[j] *= gk;
#pragma unroll
          for (int hb = 0; hb < 2; ++hb) {
            uint8_t *stg = slots + hb * 2048;
            if (h2 == 1) {  // this slot's store (piece hb of h2 = 0) has read it
              if (lane == 0) ptx::bulk_wait_read<1>();
              __syncwarp();
            }
#pragma unroll
            for (int j8 = 0; j8 < 4; ++j8)  // record layout: rotated chunks (conflict-free writes)
              *reinterpret_cast<uint4 *>(stg + rotated_chunk(lane, j8)) = pack8(x + 32 * hb + 8 * j8);
            ptx::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              ptx::bulk_s2g(recg + Rr::BI + (h2 * 2 + hb) * (128 * 64) + quarter * 2048, stg, 2048);
              ptx::bulk_commit();
            }
          }
        }
      }
    }
    ptx::fence_proxy_async_smem();  // staging slots are bulk-copy targets later
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();

    // ---- (9) M [W | U] -> cols [0, 256), M = 64 layout
    if (tid == 0) {
#pragma unroll
      for (int ks = 0; ks < kC / 16; ++ks)
        ptx::mma_bf16_ss(tmem, umma::sdesc_k(sMM, kC, ks), umma::sdesc_mn(sWU, 128, ks),
                         umma::idesc_bf16_bmn(64, 256), ks > 0);
      ptx::mma_commit(bar);
    }
    wait_mma(0x104u);
    // A's space and blocks 2-3 are free once the record stores of (8) have read
    // their slots there: fetch the next chunk's log_alpha, k, v
    if (lane == 0) ptx::bulk_wait_read<0>();
    __syncthreads();
    if (has_next) {
      if (tid == 0) issue_lkv(idx_next);
      if (tid < kC) {
        b_next = beta_of(idx_next);
        if constexpr (kRowDecay) la_next = la_row_of(idx_next);
      }
    }

    // ---- (10) token rows: Qp = Q*gamma - M W (warps 0-3), O = M U (warps 4-7).
    // M = 64 layout read as in (6): threads 0-15 hold columns 0-63 of the
    // warp's 16 rows, threads 16-31 columns 64-127.  As in (8) each warp
    // assembles contiguous record pieces in staging slots and lane 0 hands
    // them to bulk stores.  Qp: one 2 KB piece per K atom, K atom 0 in the
    // consumed W rows of block 1 and K atom 1 in place over the warp's own
    // Q*gamma rows of block 1 (each thread rewrites the 16 bytes it read);
    // both stay untouched until the next chunk's tiles.  O: two 1 KB pieces
    // per 32-column block, block hb + 1 first into block 0's consumed W rows
    // (the next chunk's q rows land there after this phase, so that store
    // is waited for here), block hb into the T tile.
    {
      const int rr = quarter * 16 + (lane & 15), side = lane >> 4, row = lane & 15;
      float x[64];
      ptx::tmem_ld32_halves<64>(t_lane + colhalf * 128, *reinterpret_cast<float(*)[32]>(x));
      ptx::tmem_ld32_halves<64>(t_lane + colhalf * 128 + 32,
                                *reinterpret_cast<float(*)[32]>(x + 32));
      ptx::tmem_ld_wait();
      if (colhalf == 0) {
        if (norm && side == 0) {  // (M W)_t0 = sum_s M_ts; Qp keeps Q*gamma there
          reinterpret_cast<float *>(nrm0 + (size_t)idx * NormRec::BYTES + NormRec::MR)[rr] = x[0];
          x[0] = 0.f;
        }
        uint8_t *const qslot = X1 + 16384 + quarter * 2048;  // K atom a at + a * 8192
        uint8_t *stg = qslot + side * 8192;
#pragma unroll
        for (int cc = 0; cc < 8; ++cc) {  // this thread's K atom is `side`
          float qg[8];
          ld_chunk(X1, kC + rr, side * 8 + cc, 128, qg);
          const float4 m0 = *reinterpret_cast<const float4 *>(gmid + side * 64 + cc * 8);
          const float4 m1 = *reinterpret_cast<const float4 *>(gmid + side * 64 + cc * 8 + 4);
          const float gm[8] = {m0.x, m0.y, m0.z, m0.w, m1.x, m1.y, m1.z, m1.w};
#pragma unroll
          for (int j = 0; j < 8; ++j) qg[j] = qg[j] * gm[j] - x[8 * cc + j];
          *reinterpret_cast<uint4 *>(stg + row * 128 + ((cc ^ (row & 7)) << 4)) = pack8(qg);
        }
        ptx::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
#pragma unroll
          for (int a = 0; a < 2; ++a)
            ptx::bulk_s2g(recg + Rr::QP + a * (kC * 128) + quarter * 2048, qslot + a * 8192, 2048);
          ptx::bulk_commit();
        }
      } else {
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const int hb = 1 - i;
          uint8_t *stg = i == 0 ? X1 + quarter * 2048 : TT + quarter * 2048;
#pragma unroll
          for (int j8 = 0; j8 < 4; ++j8)  // record layout: rotated chunks (conflict-free writes)
            *reinterpret_cast<uint4 *>(stg + side * 1024 + rotated_chunk(row, j8)) =
                pack8(x + 32 * hb + 8 * j8);
          ptx::fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
#pragma unroll
            for (int piece = 0; piece < 2; ++piece)
              ptx::bulk_s2g(recg + Rr::OI + (hb + 2 * piece) * (kC * 64) + quarter * 1024,
                            stg + piece * 1024, 1024);
            ptx::bulk_commit();
          }
        }
        if (lane == 0) ptx::bulk_wait_read<1>();  // the piece in block 0 has been read
      }
    }
    // block 0 and the TMEM columns are free again: fetch the next chunk's q
    // rows, unless a wait of this CTA gave up (then every thread leaves here)
    ptx::fence_proxy_async_smem();
    ptx::tc_fence_before();
    const int stop = __syncthreads_or(!ok);
    ptx::tc_fence_after();
    if (stop) {
      // drain (bounded) what thread 0 started: the latest row copies (the
      // next chunk's log_alpha, k, v if issued; this chunk's q), then the
      // products, before shared memory and TMEM are released
      if (tid == 0) {
        ptx::mbar_wait(lbar, (it + (has_next ? 1 : 0)) & 1, kWaitLimit);
        ptx::mbar_wait(qbar, it & 1, kWaitLimit);
        ptx::mma_commit(bar);
        ptx::mbar_wait(bar, mma_phase & 1, kWaitLimit);
      }
      break;
    }
    if (tid == 0 && has_next) issue_q(idx_next);
    l = l_next;
  }
  if (lane == 0) ptx::bulk_wait_all();  // this warp's record stores complete
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, L::TMEM_COLS);
  }
}

// n0, nseg, work: the chunk range of a pipelined call (d = 128; the d = 64
// prep always takes every chunk, n0 = 0, nseg = NC, work = total, in a fixed
// order: one CTA per SM).  ctr: the d = 128 prep's work counter, zero when
// the grid starts.  pdl (segments of a pipelined call only): the grid lets
// the next launch of the stream, its scan, be scheduled at once.  Launched
// as a programmatic dependent of the previous scan segment, a CTA starts
// while that scan still runs (its inputs and records are disjoint from the
// scan's) and waits for the scan only before it exits, so that the prep's
// completion implies the earlier scan's and the next scan segment, which
// waits for this grid, sees that scan's final state.
template <int D, int kMode, bool kRowDecay>
__global__ void __launch_bounds__(256, D == 128 ? 2 : 1)
kda_prep_kernel(const __nv_bfloat16 *__restrict__ q, const __nv_bfloat16 *__restrict__ k,
                const __nv_bfloat16 *__restrict__ v, const float *__restrict__ beta,
                const float *__restrict__ log_alpha, int alpha_mode, int T, int NC, int total,
                int n0, int nseg, int work, unsigned *ctr, uint8_t *__restrict__ ws, int rule,
                unsigned maps, int pdl) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                            ~static_cast<uintptr_t>(1023));
  if (pdl) ptx::grid_dep_launch();
  if constexpr (D == 128)
    prep_d128<kMode, kRowDecay>(q, k, v, beta, log_alpha, alpha_mode, T, NC, total, n0, nseg,
                                work, ctr, ws, sm, rule, maps);
  else
    prep_d64(q, k, v, beta, log_alpha, alpha_mode, T, NC, total, ws, sm);
  ptx::grid_dep_wait();
}

// ============================================================== scan kernel

// D = 64: the scan's two products share one M = 128 accumulator: [Ap; Qp] S
// and [Kbar^T; M] U are adjacent 64-row tiles of the record, so one group of
// eight MMAs (K = 64 each way) leaves P + Kbar^T U in lanes 0-63 (key rows)
// and o = Qp S + M U in lanes 64-127 (token rows).  Roles as in the d = 128
// scan: two state warps (thread = key row, its NB columns in registers), two
// output warps (the accumulator's lanes 64-127), a producer streaming the
// CTA's share of each record through a 3-stage ring, an issuer.  Three
// accumulators in turn let the output warps trail the state chain.
constexpr int kS64Stages = 3;
constexpr int kS64Acc = 3;
constexpr int kScan64Threads = 192;  // 2 state warps, 2 output warps, producer, issuer
template <int NB>
struct ScanSmem64 {
  using B = Rec<64>;
  static constexpr int D = 64;
  static constexpr uint32_t UT_S = B::PRE;                   // U^T block [NB rows][C]
  static constexpr uint32_t GC_S = UT_S + NB * kC * 2;       // gamma_C [D]
  static constexpr uint32_t STAGE_BYTES = GC_S + D * 4;      // Ap|Qp|Kbar^T|M, U^T block, gamma_C
  static constexpr uint32_t STAGE = align1k(STAGE_BYTES);
  static constexpr uint32_t SB = kS64Stages * STAGE;         // 2 x bf16 S [D keys][64 cols]
  static constexpr uint32_t SB_BYTES = D * 64 * 2;
  // full[kS64Stages], empty[kS64Stages], done[kS64Acc], ofree[kS64Acc]
  static constexpr uint32_t BAR = SB + 2 * SB_BYTES;
  static constexpr uint32_t TMEMP = BAR + (2 * kS64Stages + 2 * kS64Acc) * 8;
  static constexpr uint32_t ABORT = TMEMP + 4;               // CTA-wide abort word
  static constexpr uint32_t BYTES = TMEMP + 8;
  static constexpr uint32_t TMEM_COLS = 128;                 // acc[0..2], NB columns each
  static_assert(NB * kS64Acc <= (int)TMEM_COLS, "TMEM columns");
  static_assert((STAGE & 1023u) == 0 && (SB & 1023u) == 0, "operand tiles need 1024-byte alignment");
  static_assert(BYTES + 1024 <= 232448, "scan shared memory");
};

// D = 128: four roles.  A producer warp streams records through a ring of
// kStages stages.  Four state warps own S (thread = key channel, its row in
// registers as float): per chunk they write its bf16 copy (row-major, read
// MN-major by the MMA), signal the issuer, form gamma_C * S + Kbar^T U while
// the product runs, then add P = Ap S.  One issuer warp issues every MMA of
// the CTA from a single thread: P = Ap S (8 MMAs), then o = Qp S (8 MMAs)
// into one of three output accumulators.  A tcgen05.mma costs about the
// same issue time whatever its shape, and MMAs issued from several warps
// serialise with a large penalty, so one issuer keeps the pipe in order: the
// output products run while the state warps wait for P's completion and do
// their own arithmetic.  Four output warps (same TMEM lane quarters) wait
// for an output product, add M U and store o.
constexpr int kStages = 3;
constexpr int kPrefetchAhead = 3;  // scan: records prefetched into L2 this many chunks ahead of their copy
constexpr int kOutBufs = 3;
constexpr int kScan128Threads = 320;  // 4 state warps, 4 output warps, producer, issuer
// A scan CTA owns NB = 32 value columns (one block of B and O), or 64 (two
// adjacent blocks, when four CTAs per head would not fit the SMs in one
// round); the 64-column CTA has room for two record stages only.
template <int NB>
struct ScanSmem128 {
  using R = Rec<128>;
  static_assert(NB == R::BLK || NB == 2 * R::BLK, "a scan CTA owns one or two 32-column blocks");
  static constexpr int STAGES = NB == R::BLK ? kStages : 2;
  static constexpr uint32_t BI_S = R::PRE;                   // B blocks [NB / 32][128][32]
  static constexpr uint32_t OI_S = BI_S + 128 * NB * 2;      // O blocks [NB / 32][C][32]
  static constexpr uint32_t GC_S = OI_S + kC * NB * 2;       // gamma_C [128]
  static constexpr uint32_t STAGE_BYTES = GC_S + 128 * 4;
  static constexpr uint32_t NRM_S = STAGE_BYTES;             // NormRec (normalised rule only)
  static constexpr uint32_t STAGE = align1k(NRM_S + NormRec::BYTES);
  static constexpr uint32_t SB = STAGES * STAGE;             // 2 x bf16 S [128 rows][64 cols]
  // full[STAGES], empty[STAGES], mS, mO[kOutBufs], ofree[kOutBufs]
  static constexpr uint32_t BAR = SB + 2 * 128 * 64 * 2;
  static constexpr uint32_t TMEMP = BAR + (2 * STAGES + 1 + 2 * kOutBufs) * 8;
  static constexpr uint32_t ABORT = TMEMP + 4;               // CTA-wide abort word
  static constexpr uint32_t BYTES = TMEMP + 8;
  static constexpr uint32_t TMEM_COLS = NB == R::BLK ? 128 : 256;  // P | o[0] | o[1] | o[2]
  static_assert(NB * (1 + kOutBufs) <= TMEM_COLS, "TMEM columns");
  static_assert(BYTES + 1024 <= 232448, "scan shared memory");
};

// kNorm: the normalised linear-attention rule.  Its normaliser z is the
// state's column for a value of all ones (with W = 0 its update is
// z <- gamma_C z + sum_s Kbar_s): the state warps carry z_r beside row r and
// write it as column NB of the bf16 S copy, the output product runs with
// N = NB + 8, and its column NB is Qp z, to which the output warps add the
// row sum of M for the denominator.  A separate instantiation, so that the
// other rules' scan is compiled without it.
// h0 and hT may be one buffer (in-place resume): each state thread reads its
// own elements of h0 before the first chunk and writes the same elements of
// hT after the last, so neither pointer is declared __restrict__.
template <int NB, bool kNorm>
__device__ __forceinline__ void scan_d128(const float *h0, __nv_bfloat16 *__restrict__ o,
                                          float *hT, int T, int NC, int NCh, int n0,
                                          uint8_t *__restrict__ ws, uint8_t *sm) {
  constexpr int D = 128;
  constexpr uint32_t kSyncThreads = 128 + 32;  // state warps + issuer warp
  using R = Rec<128>;
  using L = ScanSmem128<NB>;
  constexpr int kStages = L::STAGES;  // record ring
  constexpr bool norm = kNorm;
  constexpr int kOW = kNorm ? NB + 8 : NB;                     // output accumulator width
  constexpr uint32_t kTmemCols = kNorm ? 256 : L::TMEM_COLS;  // P | o[0] | o[1] | o[2]
  static_assert(NB + kOutBufs * kOW <= (int)kTmemCols, "TMEM columns");
  uint64_t *full = reinterpret_cast<uint64_t *>(sm + L::BAR);
  uint64_t *empty = full + kStages;
  uint64_t *mS = empty + kStages;
  uint64_t *mO = mS + 1;
  uint64_t *ofree = mO + kOutBufs;
  uint32_t *tmem_ptr = reinterpret_cast<uint32_t *>(sm + L::TMEMP);
  uint32_t *abort_f = reinterpret_cast<uint32_t *>(sm + L::ABORT);
  WorkspaceHeader *hdr = reinterpret_cast<WorkspaceHeader *>(ws);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int bh = blockIdx.y, blk = blockIdx.x, j0 = blk * NB;
  const uint8_t *rec0 = ws + sizeof(WorkspaceHeader) + ((size_t)bh * NCh + n0) * R::BYTES;
  const uint8_t *nrm0 = ws + sizeof(WorkspaceHeader) + (size_t)gridDim.y * NCh * R::BYTES +
                        ((size_t)bh * NCh + n0) * NormRec::BYTES;
  // A wait that gives up records the error, sets the CTA's abort word and
  // makes its thread skip its later waits.  The producer then stops copying
  // and waits (bounded) for the copies it started; the issuer, which waits
  // on nothing but the state warps' named barrier, reads the abort word at
  // the end and waits (bounded) for its products before TMEM is released.
  // The other roles run out their loops, each giving up at most one wait of
  // its own: the waits on the serial path stay plain (polling the abort word
  // there cost the scan about 4 %).
  bool ok = true;

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(&full[s], 1);
      ptx::mbar_init(&empty[s], 4 + 1);  // released by each state warp and by the output warps
    }
    ptx::mbar_init(mS, 1);
    for (int b = 0; b < kOutBufs; ++b) {
      ptx::mbar_init(&mO[b], 1);
      ptx::mbar_init(&ofree[b], 1);
    }
    *abort_f = 0u;
    ptx::fence_mbar_init();
  }
  if (warp == 0) {
    ptx::tmem_alloc(tmem_ptr, kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_ptr;
  const uint32_t t_lane = tmem + ((uint32_t)((warp & 3) * 32) << 16);
  auto sb_of = [&](int chunk) { return sm + L::SB + (chunk & 1) * (128 * 64 * 2); };

  if (warp == 8) {
    // ---------------------------------------------------------- producer
    if (lane == 0) {
      int j = 0;
      for (; j < NC; ++j) {
        const int s = j % kStages;
        if (j >= kStages && ok && !ptx::mbar_wait_fast(&empty[s], ((j / kStages) - 1) & 1, kWaitLimit)) {
          ok = false;
          ptx::set_abort(abort_f);
          report_error(hdr, KDA_ERR_TIMEOUT, 0x210u);
        }
        if (!ok) break;
        uint8_t *st = sm + s * L::STAGE;
        const uint8_t *rec = rec0 + (size_t)j * R::BYTES;
        // a later record into L2 ahead of its copy, so that the copy meets L2
        // rather than DRAM latency; the Ap | Qp tile the four CTAs of a head
        // share is prefetched by one of them (all four made the scan slower)
        if (j + kPrefetchAhead < NC) {
          const uint8_t *rp = rec0 + (size_t)(j + kPrefetchAhead) * R::BYTES;
          if (blk == 0) ptx::prefetch_l2(rp, R::PRE);  // the head's shared Ap | Qp tile, once
          ptx::prefetch_l2(rp + R::BI + (size_t)blk * (128 * NB * 2), 128 * NB * 2);
          ptx::prefetch_l2(rp + R::OI + (size_t)blk * (kC * NB * 2), kC * NB * 2);
          ptx::prefetch_l2(rp + R::GC, 128 * 4);
          if (norm) ptx::prefetch_l2(nrm0 + (size_t)(j + kPrefetchAhead) * NormRec::BYTES, NormRec::BYTES);
        }
        ptx::fence_proxy_async_smem();
        ptx::mbar_arrive_expect_tx(&full[s], L::STAGE_BYTES + (norm ? NormRec::BYTES : 0u));
        if (norm)
          ptx::bulk_g2s(st + L::NRM_S, nrm0 + (size_t)j * NormRec::BYTES, NormRec::BYTES, &full[s]);
        ptx::bulk_g2s(st, rec, R::PRE, &full[s]);
        ptx::bulk_g2s(st + L::BI_S, rec + R::BI + (size_t)blk * (128 * NB * 2), 128 * NB * 2, &full[s]);
        ptx::bulk_g2s(st + L::OI_S, rec + R::OI + (size_t)blk * (kC * NB * 2), kC * NB * 2, &full[s]);
        ptx::bulk_g2s(st + L::GC_S, rec + R::GC, 128 * 4, &full[s]);
      }
      if (!ok)  // drain (bounded): the copies still in flight (j were issued)
        for (int i = j > kStages ? j - kStages : 0; i < j; ++i)
          if (!ptx::mbar_wait(&full[i % kStages], (i / kStages) & 1, kWaitLimit)) break;
    }
  } else if (warp == 9) {
    // ---------------------------------------------------------- issuer
    // The descriptors of every ring slot, formed once (a K-slice's descriptor
    // is its tile's plus a constant: shared memory addresses stay below
    // 2^18), and the loop unrolled over six chunks, the period of the 3-stage
    // record ring, the 3 output accumulators and the 2 S copies, so that
    // nothing but the MMAs sits between the hand-off and the first product.
    static_assert(6 % kStages == 0 && kOutBufs == 3, "six-chunk issuer period");
    uint64_t dAPs[kStages], dQPs[kStages], dSBs[2];
#pragma unroll
    for (int q = 0; q < kStages; ++q) {
      dAPs[q] = umma::sdesc(ptx::smem_u32(sm + q * L::STAGE + R::AP));
      dQPs[q] = umma::sdesc(ptx::smem_u32(sm + q * L::STAGE + R::QP));
    }
#pragma unroll
    for (int q = 0; q < 2; ++q) dSBs[q] = umma::sdesc_mn(ptx::smem_u32(sb_of(q)), 128, 0);
    for (int i0 = 0; i0 < NC; i0 += 6)
#pragma unroll
    for (int u = 0; u < 6; ++u) {
      const int i = i0 + u;
      if (i >= NC) break;
      const int b = u % kOutBufs;
      const uint64_t dAP = dAPs[u % kStages], dQP = dQPs[u % kStages], dSB = dSBs[u & 1];
      // bf16 S_i written and P_{i-1} read by every state thread, which have
      // also seen record i land and accumulator b freed by the output warps
      ptx::named_barrier(1, kSyncThreads);
      if (lane == 0) {
        ptx::tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks)  // P = Ap S   (S read MN-major)
          ptx::mma_bf16_ss(tmem, dAP + (uint64_t)(((ks >> 2) * D * 128 + (ks & 3) * 32) >> 4),
                           dSB + (uint64_t)(ks * 2048 >> 4), umma::idesc_bf16_bmn(128, NB), ks > 0);
        ptx::mma_commit(mS);
        const uint32_t tOc = tmem + NB + kOW * b;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks)  // o = Qp S  (and Qp z in column NB)
          ptx::mma_bf16_ss(tOc, dQP + (uint64_t)(((ks >> 2) * kC * 128 + (ks & 3) * 32) >> 4),
                           dSB + (uint64_t)(ks * 2048 >> 4), umma::idesc_bf16_bmn(64, kOW), ks > 0);
        ptx::mma_commit(&mO[b]);
      }
      __syncwarp();
    }
    if (lane == 0 && ptx::aborted(abort_f)) {  // let this thread's MMAs finish before TMEM is freed
      ptx::mma_commit(mS);
      ptx::mbar_wait(mS, NC & 1, kWaitLimit);
    }
  } else if (warp >= 4) {
    // ---------------------------------------------------------- output warps
    const int orow = (warp - 4) * 16 + lane;  // output row (M = 64 layout: lanes 32w + 0..15)
    for (int j = 0; j < NC; ++j) {
      const int b = j % kOutBufs, s = j % kStages;
      if (ok && !ptx::mbar_wait(&mO[b], (j / kOutBufs) & 1, kWaitLimit)) {
        ok = false;
        ptx::set_abort(abort_f);
        report_error(hdr, KDA_ERR_TIMEOUT, 0x221u);
      }
      if (ok && !ptx::mbar_wait_fast(&full[s], (j / kStages) & 1, kWaitLimit)) {
        ok = false;  // already complete: orders the record's bulk copy before the reads below
        ptx::set_abort(abort_f);
        report_error(hdr, KDA_ERR_TIMEOUT, 0x223u);
      }
      ptx::tc_fence_after();
      const uint32_t tO = t_lane + NB + kOW * b;
      const uint8_t *oi = sm + s * L::STAGE + L::OI_S;
      const int t = (n0 + j) * kC + orow;
      float inv_den = 1.f;
      if (norm) {  // denominator: (Qp z)_t from column NB plus the row sum of M
        float qz;
        ptx::tmem_ld1(tO + NB, qz);
        ptx::tmem_ld_wait();
        const float *nr = reinterpret_cast<const float *>(sm + s * L::STAGE + L::NRM_S);
        inv_den = 1.f / (qz + nr[NormRec::MR / 4 + (orow & (kC - 1))]);
      }
#pragma unroll
      for (int cb = 0; cb < NB; cb += 16) {
        float x[16];
        ptx::tmem_ld16(tO + cb, x);
        ptx::tmem_ld_wait();
        if (lane < 16 && t < T) {
          const int q = cb / 8;  // 16-byte chunk of the row: block q / 4, chunk q % 4
          const uint8_t *ob = oi + (q >> 2) * (kC * 64);
          const uint4 a = *reinterpret_cast<const uint4 *>(ob + rotated_chunk(orow, q & 3));
          const uint4 c2 = *reinterpret_cast<const uint4 *>(ob + rotated_chunk(orow, (q & 3) + 1));
          const uint32_t w[8] = {a.x, a.y, a.z, a.w, c2.x, c2.y, c2.z, c2.w};
          uint32_t pk[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const __nv_bfloat162 p2 = *reinterpret_cast<const __nv_bfloat162 *>(&w[e]);
            pk[e] = pack_bf16x2((x[2 * e] + __low2float(p2)) * inv_den,
                                (x[2 * e + 1] + __high2float(p2)) * inv_den);
          }
          uint4 *dst = reinterpret_cast<uint4 *>(o + ((size_t)bh * T + t) * D + j0 + cb);
          dst[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
          dst[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
        }
      }
      ptx::tc_fence_before();
      ptx::named_barrier(2, 128);  // all output rows of chunk j read
      if (tid == 128) {
        ptx::mbar_arrive(&ofree[b]);
        ptx::mbar_arrive(&empty[s]);
      }
    }
  } else {
    // ---------------------------------------------------------- state warps
    // Thread r keeps row r of S (key channel r, this CTA's NB value columns)
    // in registers as float.  Per chunk: its bf16 copy goes to the operand
    // buffer (free again: the products that read it two chunks ago completed
    // before the last P), the issuer is told, each thread forms
    // gamma_C S + B while the product runs, then S <- that + P.
    const int r = tid;  // key channel = TMEM lane
    const uint32_t tP = t_lane;
    float zr = 0.f;     // normalised rule: z_r (zero initial state)
    float sr[NB];
    {
      const size_t s0 = (size_t)bh * D * D + (size_t)r * D + j0;
#pragma unroll
      for (int j = 0; j < NB; ++j) sr[j] = h0 ? h0[s0 + j] : 0.f;
    }
    for (int i = 0; i < NC; ++i) {
      const int s = i % kStages;
      const uint8_t *st = sm + s * L::STAGE;
      uint8_t *sb = sb_of(i);
#pragma unroll
      for (int c8 = 0; c8 < NB / 8; ++c8) st_chunk(sb, r, c8, 128, sr + 8 * c8);
      if (norm) {
        const float zc[8] = {zr, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        st_chunk(sb, r, NB / 8, 128, zc);
      }
      ptx::fence_proxy_async_smem();
      ptx::tc_fence_before();
      // the checks the issuer's products need, made here where they are off
      // its serial path: record i landed (every state thread reads its B and
      // gamma_C below anyway), accumulator (i mod 3) read by the output warps
      // (chunk i - 3)
      if (ok && !ptx::mbar_wait_fast(&full[s], (i / kStages) & 1, kWaitLimit)) {
        ok = false;
        ptx::set_abort(abort_f);
        report_error(hdr, KDA_ERR_TIMEOUT, 0x204u);
      }
      if (r == 0) {
        if (i >= kOutBufs && ok &&
            !ptx::mbar_wait_fast(&ofree[i % kOutBufs], ((i / kOutBufs) - 1) & 1, kWaitLimit)) {
          ok = false;
          ptx::set_abort(abort_f);
          report_error(hdr, KDA_ERR_TIMEOUT, 0x222u);
        }
      }
      __syncwarp();
      // two-stage ring: stage i - 1 for the state side here, by each state
      // warp (released at the end of its chunk, as the three-stage ring does,
      // the 64-column scan measured 0.365 -> 0.379 ms on Gated DeltaNet)
      if (kStages == 2 && lane == 0 && i > 0) ptx::mbar_arrive(&empty[(i - 1) % kStages]);
      ptx::named_arrive(1, kSyncThreads);
      {  // gamma_C S + B while the product runs
        const float gam = reinterpret_cast<const float *>(st + L::GC_S)[r];
        if (norm)
          zr = gam * zr + reinterpret_cast<const float *>(st + L::NRM_S)[NormRec::KS / 4 + r];
#pragma unroll
        for (int q4 = 0; q4 < NB / 8; ++q4) {
          const uint4 a = *reinterpret_cast<const uint4 *>(st + L::BI_S + (q4 >> 2) * (128 * 64) +
                                                           rotated_chunk(r, q4 & 3));
          const uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const __nv_bfloat162 p2 = *reinterpret_cast<const __nv_bfloat162 *>(&w[e]);
            sr[8 * q4 + 2 * e] = gam * sr[8 * q4 + 2 * e] + __low2float(p2);
            sr[8 * q4 + 2 * e + 1] = gam * sr[8 * q4 + 2 * e + 1] + __high2float(p2);
          }
        }
      }
      if (ok && !ptx::mbar_wait(mS, i & 1, kWaitLimit)) {
        ok = false;
        ptx::set_abort(abort_f);
        report_error(hdr, KDA_ERR_TIMEOUT, 0x201u);
      }
      ptx::tc_fence_after();
      {
        float x[NB];
#pragma unroll
        for (int c = 0; c < NB; c += 32)
          ptx::tmem_ld32(tP + c, *reinterpret_cast<float(*)[32]>(x + c));
        ptx::tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < NB; ++j) sr[j] += x[j];
      }
      // three-stage ring: stage s for the state side, by each state warp: its
      // lanes have read their B rows and seen P_i, the stage's last state-side
      // product, complete (here rather than after the next chunk's hand-off:
      // the producer's next copy starts that much earlier, 1.60 -> 1.58 ms)
      if (kStages == 3) {
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&empty[s]);
      }
    }
    if (hT) {
      float4 *dst = reinterpret_cast<float4 *>(hT + (size_t)bh * D * D + (size_t)r * D + j0);
#pragma unroll
      for (int j4 = 0; j4 < NB / 4; ++j4)
        dst[j4] = make_float4(sr[4 * j4], sr[4 * j4 + 1], sr[4 * j4 + 2], sr[4 * j4 + 3]);
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

template <int NB>
__device__ __forceinline__ void scan_d64(const float *h0, __nv_bfloat16 *__restrict__ o,
                                         float *hT, int T, int NC, int NCh, int n0,
                                         uint8_t *__restrict__ ws, uint8_t *sm) {
  constexpr int D = 64;
  constexpr uint32_t kSyncThreads = 64 + 32;  // state warps + issuer warp
  using R = Rec<64>;
  using L = ScanSmem64<NB>;
  uint64_t *full = reinterpret_cast<uint64_t *>(sm + L::BAR);
  uint64_t *empty = full + kS64Stages;
  uint64_t *done = empty + kS64Stages;
  uint64_t *ofree = done + kS64Acc;
  uint32_t *tmem_ptr = reinterpret_cast<uint32_t *>(sm + L::TMEMP);
  uint32_t *abort_f = reinterpret_cast<uint32_t *>(sm + L::ABORT);
  WorkspaceHeader *hdr = reinterpret_cast<WorkspaceHeader *>(ws);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int bh = blockIdx.y, blk = blockIdx.x, j0 = blk * NB;
  const uint8_t *rec0 = ws + sizeof(WorkspaceHeader) + ((size_t)bh * NCh + n0) * R::BYTES;
  // after a failed wait, as in the d = 128 scan: the abort word is set, the
  // producer stops copying and drains its copies, the issuer drains its
  // products, the other roles run out their loops without waiting
  bool ok = true;
  auto fail = [&](unsigned where) {
    ok = false;
    ptx::set_abort(abort_f);
    report_error(hdr, KDA_ERR_TIMEOUT, where);
  };

  if (tid == 0) {
    for (int s = 0; s < kS64Stages; ++s) {
      ptx::mbar_init(&full[s], 1);
      ptx::mbar_init(&empty[s], 2);  // lane 0 of each state warp, once its products completed
    }
    for (int b = 0; b < kS64Acc; ++b) {
      ptx::mbar_init(&done[b], 1);
      ptx::mbar_init(&ofree[b], 2);  // lane 0 of each output warp
    }
    *abort_f = 0u;
    ptx::fence_mbar_init();
  }
  if (warp == 0) {
    ptx::tmem_alloc(tmem_ptr, L::TMEM_COLS);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_ptr;
  const uint32_t t_lane = tmem + ((uint32_t)((warp & 3) * 32) << 16);
  auto sb_of = [&](int chunk) { return sm + L::SB + (chunk & 1) * L::SB_BYTES; };

  if (warp == 4) {
    // ---------------------------------------------------------- producer
    if (lane == 0) {
      int j = 0;
      for (; j < NC; ++j) {
        const int s = j % kS64Stages;
        if (j >= kS64Stages && ok &&
            !ptx::mbar_wait_fast(&empty[s], ((j / kS64Stages) - 1) & 1, kWaitLimit))
          fail(0x410u);
        if (!ok) break;
        if (j + kPrefetchAhead < NC) {  // a later record into L2 (the shared part by one CTA)
          const uint8_t *rp = rec0 + (size_t)(j + kPrefetchAhead) * R::BYTES;
          if (blk == 0) ptx::prefetch_l2(rp, R::PRE);
          ptx::prefetch_l2(rp + R::UT + (size_t)j0 * (kC * 2), NB * kC * 2);
          ptx::prefetch_l2(rp + R::GC, D * 4);
        }
        uint8_t *st = sm + s * L::STAGE;
        const uint8_t *rec = rec0 + (size_t)j * R::BYTES;
        ptx::fence_proxy_async_smem();
        ptx::mbar_arrive_expect_tx(&full[s], L::STAGE_BYTES);
        ptx::bulk_g2s(st, rec, R::PRE, &full[s]);
        ptx::bulk_g2s(st + L::UT_S, rec + R::UT + (size_t)j0 * (kC * 2), NB * kC * 2, &full[s]);
        ptx::bulk_g2s(st + L::GC_S, rec + R::GC, D * 4, &full[s]);
      }
      if (!ok)  // drain (bounded): the copies still in flight (j were issued)
        for (int i = j > kS64Stages ? j - kS64Stages : 0; i < j; ++i)
          if (!ptx::mbar_wait(&full[i % kS64Stages], (i / kS64Stages) & 1, kWaitLimit)) break;
    }
  } else if (warp == 5) {
    // ---------------------------------------------------------- issuer
    uint64_t dAs[kS64Stages], dKs[kS64Stages], dUs[kS64Stages], dSBs[2];
#pragma unroll
    for (int q = 0; q < kS64Stages; ++q) {
      uint8_t *st = sm + q * L::STAGE;
      dAs[q] = umma::sdesc(ptx::smem_u32(st + R::AP));   // [Ap; Qp]     128 rows, K = D
      dKs[q] = umma::sdesc(ptx::smem_u32(st + R::KBT));  // [Kbar^T; M]  128 rows, K = C
      dUs[q] = umma::sdesc(ptx::smem_u32(st + L::UT_S)); // U^T block    NB rows, K = C
    }
#pragma unroll
    for (int q = 0; q < 2; ++q) dSBs[q] = umma::sdesc_mn(ptx::smem_u32(sb_of(q)), D, 0);
    static_assert(kS64Stages == 3 && kS64Acc == 3, "six-chunk issuer period");
    for (int i0 = 0; i0 < NC; i0 += 6)
#pragma unroll
    for (int u = 0; u < 6; ++u) {
      const int i = i0 + u;
      if (i >= NC) break;
      const int b = u % kS64Acc;
      const uint64_t dA = dAs[u % kS64Stages], dK = dKs[u % kS64Stages],
                     dU = dUs[u % kS64Stages], dSB = dSBs[u & 1];
      ptx::named_barrier(1, kSyncThreads);  // S_i written, record i landed, acc b free
      if (lane == 0) {
        ptx::tc_fence_after();
        const uint32_t tA = tmem + NB * b;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks)  // [Ap; Qp] S   (S read MN-major)
          ptx::mma_bf16_ss(tA, dA + (uint64_t)((ks * 32) >> 4), dSB + (uint64_t)(ks * 2048 >> 4),
                           umma::idesc_bf16_bmn(128, NB), ks > 0);
#pragma unroll
        for (int ks = 0; ks < kC / 16; ++ks)  // + [Kbar^T; M] U
          ptx::mma_bf16_ss(tA, dK + (uint64_t)((ks * 32) >> 4), dU + (uint64_t)((ks * 32) >> 4),
                           umma::idesc_bf16(128, NB), 1);
        ptx::mma_commit(&done[b]);
      }
      __syncwarp();
    }
    if (lane == 0 && ptx::aborted(abort_f)) {  // let this thread's MMAs finish before TMEM is freed
      ptx::mma_commit(&done[0]);
      ptx::mbar_wait(&done[0], ((NC + kS64Acc - 1) / kS64Acc) & 1, kWaitLimit);
    }
  } else if (warp >= 2) {
    // ---------------------------------------------------------- output warps
    const int row = (warp - 2) * 32 + lane;  // token row of the chunk (accumulator lane 64 + row)
    for (int j = 0; j < NC; ++j) {
      const int b = j % kS64Acc;
      if (ok && !ptx::mbar_wait(&done[b], (j / kS64Acc) & 1, kWaitLimit)) fail(0x421u);
      ptx::tc_fence_after();
      float x[NB];
      ptx::tmem_ld32(t_lane + NB * b, *reinterpret_cast<float(*)[32]>(x));
      ptx::tmem_ld_wait();
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&ofree[b]);
      const int t = (n0 + j) * kC + row;
      if (t < T) {
        uint4 *dst = reinterpret_cast<uint4 *>(o + ((size_t)bh * T + t) * D + j0);
#pragma unroll
        for (int c8 = 0; c8 < NB / 8; ++c8) {
          const float *v8 = x + 8 * c8;
          dst[c8] = make_uint4(pack_bf16x2(v8[0], v8[1]), pack_bf16x2(v8[2], v8[3]),
                               pack_bf16x2(v8[4], v8[5]), pack_bf16x2(v8[6], v8[7]));
        }
      }
    }
  } else {
    // ---------------------------------------------------------- state warps
    const int r = tid;  // key row = accumulator lane
    float sr[NB];
#pragma unroll
    for (int j = 0; j < NB; ++j) sr[j] = 0.f;
    if (h0) {
      const float4 *src = reinterpret_cast<const float4 *>(h0 + (size_t)bh * D * D + (size_t)r * D + j0);
#pragma unroll
      for (int j4 = 0; j4 < NB / 4; ++j4) {
        const float4 a = src[j4];
        sr[4 * j4] = a.x; sr[4 * j4 + 1] = a.y; sr[4 * j4 + 2] = a.z; sr[4 * j4 + 3] = a.w;
      }
    }
    for (int i = 0; i < NC; ++i) {
      const int s = i % kS64Stages, b = i % kS64Acc;
      const uint8_t *st = sm + s * L::STAGE;
      uint8_t *sb = sb_of(i);
#pragma unroll
      for (int c8 = 0; c8 < NB / 8; ++c8) st_chunk(sb, r, c8, D, sr + 8 * c8);
      ptx::fence_proxy_async_smem();
      ptx::tc_fence_before();
      // record i landed (gamma_C is read below); accumulator b read by the
      // output warps (chunk i - 3)
      if (ok && !ptx::mbar_wait_fast(&full[s], (i / kS64Stages) & 1, kWaitLimit)) fail(0x404u);
      if (r == 0 && i >= kS64Acc && ok &&
          !ptx::mbar_wait_fast(&ofree[b], ((i / kS64Acc) - 1) & 1, kWaitLimit))
        fail(0x422u);
      __syncwarp();
      ptx::named_arrive(1, kSyncThreads);
      const float gam = reinterpret_cast<const float *>(st + L::GC_S)[r];
#pragma unroll
      for (int j = 0; j < NB; ++j) sr[j] *= gam;  // gamma_C S while the products run
      if (ok && !ptx::mbar_wait(&done[b], (i / kS64Acc) & 1, kWaitLimit)) fail(0x401u);
      ptx::tc_fence_after();
      {
        float x[NB];
        ptx::tmem_ld32(t_lane + NB * b, *reinterpret_cast<float(*)[32]>(x));
        ptx::tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < NB; ++j) sr[j] += x[j];  // + Ap S + Kbar^T U
      }
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&empty[s]);  // the products and this warp's reads are done
    }
    if (hT) {
      float4 *dst = reinterpret_cast<float4 *>(hT + (size_t)bh * D * D + (size_t)r * D + j0);
#pragma unroll
      for (int j4 = 0; j4 < NB / 4; ++j4)
        dst[j4] = make_float4(sr[4 * j4], sr[4 * j4 + 1], sr[4 * j4 + 2], sr[4 * j4 + 3]);
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, L::TMEM_COLS);
  }
}

// D = 128, one CTA per (batch, head) holding all 128 value columns ("wide"
// scan, KDA_PATH_TENSOR_WIDE_SCAN).  The value-column split above gives a
// head four CTAs, each issuing the same sixteen MMAs per chunk on a 32-column
// slice; this CTA issues the sixteen on N = 128 and so needs a quarter of the
// CTAs (one round where the split needs several when heads outnumber a
// quarter of the SMs), but streams each whole 98.8 KB record through one SM.
// Measured on Gated DeltaNet (8 x 16 heads x 8192 tokens) it matched the
// split scan (0.442 against 0.434 ms: the records' HBM traffic bounds both),
// so the automatic choice stays with the split scan.  Roles:
//  - eight state warps: warp w owns key rows 32 (w mod 4) .. +31 (its TMEM
//    lane quarter) and value columns 64 (w / 4) .. +63, each thread one row
//    of 64 columns in registers as float;
//  - two output warps, each thread one token row x 128 columns (the output
//    product is issued with M = 128: the 64 rows past the chunk's read the
//    bytes that follow the Qp tile and land in TMEM lanes 64-127, which
//    nothing reads; so two lane quarters hold the rows and two warps suffice);
//  - a producer warp streaming the MMA operands Ap | Qp through a 3-stage
//    ring with gamma_C beside them, and prefetching whole records into L2
//    three chunks ahead;
//  - an issuer warp: P = Ap S (8 MMAs, M = 128, N = 128), then o = Qp S
//    (8 MMAs, M = 128 as above, N = 128) into one of two output accumulators.
// The additive terms B = Kbar^T U (state warps) and O = M U (output warps)
// are not staged: each thread loads its 128-byte slice from L2 at the start
// of the chunk that adds it (the state warps before they hand S over, the
// output warps before they wait for the product), which keeps the ring, the
// two bf16 copies of S and 512 TMEM columns inside one SM.
constexpr int kWStages = 3;
constexpr int kWOutBufs = 2;
constexpr int kWideThreads = 384;  // 8 state warps, 2 output warps, producer, issuer
struct ScanWideSmem {
  using R = Rec<128>;
  static constexpr uint32_t STAGE = R::PRE;                    // Ap | Qp (48 KB)
  static_assert((STAGE & 1023u) == 0, "stage alignment");
  static constexpr uint32_t SB = kWStages * STAGE;             // 2 x bf16 S [128 keys][128 values]
  static constexpr uint32_t SB_BYTES = 128 * 128 * 2;
  static constexpr uint32_t GC = SB + 2 * SB_BYTES;            // gamma_C [kWStages][128] float
  // full[kWStages], empty[kWStages], mS, mO[kWOutBufs], ofree[kWOutBufs]
  static constexpr uint32_t BAR = GC + kWStages * 128 * 4;
  static constexpr uint32_t TMEMP = BAR + (2 * kWStages + 1 + 2 * kWOutBufs) * 8;
  static constexpr uint32_t ABORT = TMEMP + 4;                 // CTA-wide abort word
  static constexpr uint32_t BYTES = TMEMP + 8;
  static constexpr uint32_t TMEM_COLS = 512;                   // P | o[0] | o[1], 128 each
  static_assert(128 * (1 + kWOutBufs) <= (int)TMEM_COLS, "TMEM columns");
  static_assert(BYTES + 1024 <= 232448, "wide scan shared memory");
};

// 32 * n bf16 of row r of a [4][rows][32] rotated block array (B or O of a
// record), blocks blk0 .. blk0 + n - 1 (columns 32 blk0 ..), as 16-byte loads
// from L2.
template <int n>
__device__ __forceinline__ void load_row_blocks(const uint8_t *blocks, int rows, int r, int blk0,
                                                uint4 (&u)[4 * n]) {
#pragma unroll
  for (int b2 = 0; b2 < n; ++b2)
#pragma unroll
    for (int q = 0; q < 4; ++q)
      u[4 * b2 + q] = __ldg(reinterpret_cast<const uint4 *>(
          blocks + (size_t)(blk0 + b2) * rows * 64 + rotated_chunk(r, q)));
}

__device__ __forceinline__ void scan_wide_d128(const float *h0, __nv_bfloat16 *__restrict__ o,
                                               float *hT, int T, int NC, int NCh, int n0,
                                               uint8_t *__restrict__ ws, uint8_t *sm) {
  constexpr int D = 128;
  constexpr uint32_t kSyncThreads = 256 + 32;  // state warps + issuer warp
  using R = Rec<128>;
  using L = ScanWideSmem;
  uint64_t *full = reinterpret_cast<uint64_t *>(sm + L::BAR);
  uint64_t *empty = full + kWStages;
  uint64_t *mS = empty + kWStages;
  uint64_t *mO = mS + 1;
  uint64_t *ofree = mO + kWOutBufs;
  uint32_t *tmem_ptr = reinterpret_cast<uint32_t *>(sm + L::TMEMP);
  uint32_t *abort_f = reinterpret_cast<uint32_t *>(sm + L::ABORT);
  const float *gcr = reinterpret_cast<const float *>(sm + L::GC);
  WorkspaceHeader *hdr = reinterpret_cast<WorkspaceHeader *>(ws);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int bh = blockIdx.x;
  const uint8_t *rec0 = ws + sizeof(WorkspaceHeader) + ((size_t)bh * NCh + n0) * R::BYTES;
  // After a failed wait: the abort word is set and the thread skips its later
  // waits; the producer stops copying and drains its copies, the issuer
  // drains its products before TMEM is released (as in the split scan).
  bool ok = true;
  auto fail = [&](unsigned where) {
    ok = false;
    ptx::set_abort(abort_f);
    report_error(hdr, KDA_ERR_TIMEOUT, where);
  };

  if (tid == 0) {
    for (int s = 0; s < kWStages; ++s) {
      ptx::mbar_init(&full[s], 1);
      ptx::mbar_init(&empty[s], 8 + 1);  // released by each state warp and by the output warps
    }
    ptx::mbar_init(mS, 1);
    for (int b = 0; b < kWOutBufs; ++b) {
      ptx::mbar_init(&mO[b], 1);
      ptx::mbar_init(&ofree[b], 1);
    }
    *abort_f = 0u;
    ptx::fence_mbar_init();
  }
  if (warp == 0) {
    ptx::tmem_alloc(tmem_ptr, L::TMEM_COLS);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_ptr;
  const uint32_t t_lane = tmem + ((uint32_t)((warp & 3) * 32) << 16);
  auto sb_of = [&](int chunk) { return sm + L::SB + (chunk & 1) * L::SB_BYTES; };

  if (warp == 10) {
    // ---------------------------------------------------------- producer
    if (lane == 0) {
      int j = 0;
      for (; j < NC; ++j) {
        const int s = j % kWStages;
        if (j >= kWStages && ok &&
            !ptx::mbar_wait_fast(&empty[s], ((j / kWStages) - 1) & 1, kWaitLimit))
          fail(0x310u);
        if (!ok) break;
        // whole records into L2 three chunks ahead: the stage copies and the
        // state and output warps' loads of B and O then meet L2, not DRAM
        if (j + kPrefetchAhead < NC)
          ptx::prefetch_l2(rec0 + (size_t)(j + kPrefetchAhead) * R::BYTES, R::BYTES);
        const uint8_t *rec = rec0 + (size_t)j * R::BYTES;
        ptx::fence_proxy_async_smem();
        ptx::mbar_arrive_expect_tx(&full[s], R::PRE + 128 * 4);
        ptx::bulk_g2s(sm + s * L::STAGE, rec, R::PRE, &full[s]);
        ptx::bulk_g2s(sm + L::GC + s * 512, rec + R::GC, 128 * 4, &full[s]);
      }
      if (!ok)  // drain (bounded): the copies still in flight (j were issued)
        for (int i = j > kWStages ? j - kWStages : 0; i < j; ++i)
          if (!ptx::mbar_wait(&full[i % kWStages], (i / kWStages) & 1, kWaitLimit)) break;
    }
  } else if (warp == 11) {
    // ---------------------------------------------------------- issuer
    uint64_t dAPs[kWStages], dQPs[kWStages], dSBs[2];
#pragma unroll
    for (int q = 0; q < kWStages; ++q) {
      dAPs[q] = umma::sdesc(ptx::smem_u32(sm + q * L::STAGE + R::AP));
      dQPs[q] = umma::sdesc(ptx::smem_u32(sm + q * L::STAGE + R::QP));
    }
#pragma unroll
    for (int q = 0; q < 2; ++q) dSBs[q] = umma::sdesc_mn(ptx::smem_u32(sb_of(q)), 128, 0);
    static_assert(kWStages == 3 && kWOutBufs == 2, "six-chunk issuer period");
    for (int i0 = 0; i0 < NC; i0 += 6)
#pragma unroll
    for (int u = 0; u < 6; ++u) {
      const int i = i0 + u;
      if (i >= NC) break;
      const int b = u % kWOutBufs;
      const uint64_t dAP = dAPs[u % kWStages], dQP = dQPs[u % kWStages], dSB = dSBs[u & 1];
      ptx::named_barrier(1, kSyncThreads);  // S_i written, record i landed, o[b] free
      if (lane == 0) {
        ptx::tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks)  // P = Ap S   (S read MN-major, N = 128)
          ptx::mma_bf16_ss(tmem, dAP + (uint64_t)(((ks >> 2) * D * 128 + (ks & 3) * 32) >> 4),
                           dSB + (uint64_t)(ks * 2048 >> 4), umma::idesc_bf16_bmn(128, D), ks > 0);
        ptx::mma_commit(mS);
        const uint32_t tOc = tmem + D + D * b;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks)  // o = Qp S  (M = 128: rows 64-127 unused)
          ptx::mma_bf16_ss(tOc, dQP + (uint64_t)(((ks >> 2) * kC * 128 + (ks & 3) * 32) >> 4),
                           dSB + (uint64_t)(ks * 2048 >> 4), umma::idesc_bf16_bmn(128, D), ks > 0);
        ptx::mma_commit(&mO[b]);
      }
      __syncwarp();
    }
    if (lane == 0 && ptx::aborted(abort_f)) {  // let this thread's MMAs finish before TMEM is freed
      ptx::mma_commit(mS);
      ptx::mbar_wait(mS, NC & 1, kWaitLimit);
    }
  } else if (warp >= 8) {
    // ---------------------------------------------------------- output warps
    // warp 8 + w reads TMEM lane quarter w: token rows 32 w + lane
    const int row = (warp - 8) * 32 + lane;
    const uint8_t *orec = rec0 + R::OI;
    for (int j = 0; j < NC; ++j, orec += R::BYTES) {
      const int b = j % kWOutBufs, s = j % kWStages;
      uint4 Oc[8];  // O of this row, columns 0-63, from L2, loaded while the product runs
      load_row_blocks<2>(orec, kC, row, 0, Oc);
      if (ok && !ptx::mbar_wait(&mO[b], (j / kWOutBufs) & 1, kWaitLimit)) fail(0x321u);
      ptx::tc_fence_after();
      const uint32_t tO = t_lane + D + D * b;
      const int t = (n0 + j) * kC + row;
#pragma unroll
      for (int c = 0; c < 4; ++c) {  // 32-column block c of the row
        if (c == 2) load_row_blocks<2>(orec, kC, row, 2, Oc);  // columns 64-127
        float x[32];
        ptx::tmem_ld32(tO + 32 * c, x);
        ptx::tmem_ld_wait();
        uint32_t pk[16];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint4 a = Oc[4 * (c & 1) + q];
          const uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const __nv_bfloat162 p2 = *reinterpret_cast<const __nv_bfloat162 *>(&w[e]);
            pk[4 * q + e] = pack_bf16x2(x[8 * q + 2 * e] + __low2float(p2),
                                        x[8 * q + 2 * e + 1] + __high2float(p2));
          }
        }
        if (t < T) {
          uint4 *dst = reinterpret_cast<uint4 *>(o + ((size_t)bh * T + t) * D + 32 * c);
#pragma unroll
          for (int q = 0; q < 4; ++q)
            dst[q] = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
        }
      }
      ptx::tc_fence_before();
      ptx::named_barrier(2, 64);  // all output rows of chunk j read from TMEM
      if (tid == 256) {
        ptx::mbar_arrive(&ofree[b]);
        ptx::mbar_arrive(&empty[s]);  // Qp of stage s was read by the output product
      }
    }
  } else {
    // ---------------------------------------------------------- state warps
    const int r = (warp & 3) * 32 + lane, half = warp >> 2;  // key row, column half
    const uint32_t tP = t_lane + 64 * half;
    float sr[64];
#pragma unroll
    for (int j = 0; j < 64; ++j) sr[j] = 0.f;
    if (h0) {
      const float4 *src = reinterpret_cast<const float4 *>(h0 + (size_t)bh * D * D + (size_t)r * D +
                                                           64 * half);
#pragma unroll
      for (int j4 = 0; j4 < 16; ++j4) {
        const float4 a = src[j4];
        sr[4 * j4] = a.x; sr[4 * j4 + 1] = a.y; sr[4 * j4 + 2] = a.z; sr[4 * j4 + 3] = a.w;
      }
    }
    for (int i = 0; i < NC; ++i) {
      const int s = i % kWStages;
      uint8_t *sb = sb_of(i);
      uint4 Bc[8];  // this chunk's B row slice, from L2 (used after the hand-off)
      load_row_blocks<2>(rec0 + (size_t)i * R::BYTES + R::BI, 128, r, 2 * half, Bc);
#pragma unroll
      for (int c8 = 0; c8 < 8; ++c8) st_chunk(sb, r, 8 * half + c8, 128, sr + 8 * c8);
      ptx::fence_proxy_async_smem();
      ptx::tc_fence_before();
      // record i landed (gamma_C is read below), output accumulator (i mod 2)
      // read by the output warps (chunk i - 2); stage i - 1 released by each
      // state warp (its lanes read their gamma_C of chunk i - 1 and saw
      // P_{i-1}, the stage's last state-side product, complete)
      if (ok && !ptx::mbar_wait_fast(&full[s], (i / kWStages) & 1, kWaitLimit)) fail(0x304u);
      if (tid == 0 && i >= kWOutBufs && ok &&
          !ptx::mbar_wait_fast(&ofree[i % kWOutBufs], ((i / kWOutBufs) - 1) & 1, kWaitLimit))
        fail(0x322u);
      __syncwarp();
      if (lane == 0 && i > 0) ptx::mbar_arrive(&empty[(i - 1) % kWStages]);
      ptx::named_arrive(1, kSyncThreads);
      {  // gamma_C S + B while the product runs
        const float gam = gcr[s * 128 + r];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const uint32_t w[4] = {Bc[q].x, Bc[q].y, Bc[q].z, Bc[q].w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const __nv_bfloat162 p2 = *reinterpret_cast<const __nv_bfloat162 *>(&w[e]);
            sr[8 * q + 2 * e] = gam * sr[8 * q + 2 * e] + __low2float(p2);
            sr[8 * q + 2 * e + 1] = gam * sr[8 * q + 2 * e + 1] + __high2float(p2);
          }
        }
      }
      if (ok && !ptx::mbar_wait(mS, i & 1, kWaitLimit)) fail(0x301u);
      ptx::tc_fence_after();
#pragma unroll
      for (int c4 = 0; c4 < 4; ++c4) {
        float x[16];
        ptx::tmem_ld16(tP + 16 * c4, x);
        ptx::tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 16; ++j) sr[16 * c4 + j] += x[j];
      }
    }
    if (hT) {
      float4 *dst = reinterpret_cast<float4 *>(hT + (size_t)bh * D * D + (size_t)r * D + 64 * half);
#pragma unroll
      for (int j4 = 0; j4 < 16; ++j4)
        dst[j4] = make_float4(sr[4 * j4], sr[4 * j4 + 1], sr[4 * j4 + 2], sr[4 * j4 + 3]);
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, L::TMEM_COLS);
  }
}

// The scans take chunks n0 .. n0 + NC - 1 of each head (NCh chunks per head
// in the workspace): all of them in one call, or one segment of a pipelined
// call, where h0 is the state after chunk n0 - 1 (hT of the previous segment,
// possibly the same buffer) and hT the state after the segment.  Launched as
// a programmatic dependent of the prep segment that writes its records, a
// scan waits for its own prep (and through it for the previous scan segment)
// before it reads; with pdl set (every scan segment but the last) it lets the
// next prep segment be scheduled at once.
__global__ void __launch_bounds__(kWideThreads, 1)
kda_scan_wide_kernel(const float *h0, __nv_bfloat16 *__restrict__ o, float *hT, int T, int NC,
                     int NCh, int n0, uint8_t *__restrict__ ws, int pdl) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                            ~static_cast<uintptr_t>(1023));
  if (pdl) ptx::grid_dep_launch();
  ptx::grid_dep_wait();
  scan_wide_d128(h0, o, hT, T, NC, NCh, n0, ws, sm);
}

template <int D, int NB, bool kNorm>
__global__ void __launch_bounds__(kScan128Threads, 1)
kda_scan_kernel(const float *h0, __nv_bfloat16 *__restrict__ o, float *hT, int T, int NC,
                int NCh, int n0, uint8_t *__restrict__ ws, int pdl) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                            ~static_cast<uintptr_t>(1023));
  if (pdl) ptx::grid_dep_launch();
  ptx::grid_dep_wait();
  if constexpr (D == 128)
    scan_d128<NB, kNorm>(h0, o, hT, T, NC, NCh, n0, ws, sm);
  else
    scan_d64<NB>(h0, o, hT, T, NC, NCh, n0, ws, sm);
}

// ============================================================== launch

template <int D>
constexpr int scan_nb() { return 32; }

int sm_count() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return 0;
  return sms;
}

// Launch with or without programmatic stream serialization (see the prep and
// scan kernels for what each side waits for).
template <typename... KArgs, typename... Args>
cudaError_t launch_k(void (*kern)(KArgs...), dim3 grid, int threads, uint32_t smem,
                     cudaStream_t st, bool pdl, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3((unsigned)threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

// The state between the segments of a pipelined call when the caller wants
// no final state: after the records and their normaliser sums.
float *segment_state(uint8_t *ws, int BH, int NC) {
  return reinterpret_cast<float *>(ws + sizeof(WorkspaceHeader) +
                                   (size_t)BH * NC * (Rec<128>::BYTES + NormRec::BYTES));
}
// The d = 128 prep's work counters (one per segment), after the states;
// zeroed on the stream at the start of every call.
constexpr int kMaxSegments = 16;
constexpr size_t kClaimBytes = 256;
static_assert(kMaxSegments * sizeof(unsigned) <= kClaimBytes, "claim area");
unsigned *claim_area(uint8_t *ws, int BH, int NC) {
  return reinterpret_cast<unsigned *>(reinterpret_cast<uint8_t *>(segment_state(ws, BH, NC)) +
                                      (size_t)BH * 128 * 128 * sizeof(float));
}

// One prep launch and one scan launch per segment of G (G = 1: the whole
// sequence, prep then scan).  Pipelined (G > 1, d = 128): segment g's prep
// (all heads, chunks [g s, g s + s)) then its scan; every launch after the
// first is a programmatic dependent of the one before, so scan g (the
// one-CTA-per-head scan, on BH SMs) runs beside prep g + 1 (two CTAs per SM
// on the other SMs).  The last segment's scan, with no prep beside it, is
// the split scan.
template <int D>
kda_status launch_d(const void *q, const void *k, const void *v, const float *beta,
                    const float *log_alpha, const float *h0, void *o, float *hT, int BH, int T,
                    kda_alpha_mode am, uint8_t *ws, cudaStream_t st, LaunchTimer &timer,
                    int rule, unsigned maps, bool wide, int G) {
  constexpr int NB = scan_nb<D>();
  const int NC = (T + kC - 1) / kC;
  const int sms = sm_count();
  if (sms <= 0) return KDA_ERR_CUDA;
  // d = 128: 64 value columns per scan CTA when four CTAs per head would
  // take more than one round of the SMs (not the normalised rule)
  const bool nb64 = D == 128 && rule != KDA_RULE_LINEAR_NORM && (long long)BH * (D / NB) > sms;
  const int scan_nbv = nb64 ? 2 * NB : NB;
  const uint32_t prep_smem = (D == 128 ? PrepSmem128::BYTES : PrepSmem64::BYTES) + 1024;
  const uint32_t scan_smem =
      (D == 128 ? (nb64 ? ScanSmem128<2 * NB>::BYTES : ScanSmem128<NB>::BYTES)
                : ScanSmem64<NB>::BYTES) + 1024;
  auto prep = kda_prep_kernel<D, 0, false>;
  if constexpr (D == 128) {
    const bool row = am != KDA_ALPHA_CHANNEL;  // scalar or no decay: one factor per token
    if (rule != KDA_RULE_DELTA)
      prep = row ? kda_prep_kernel<D, 2, true> : kda_prep_kernel<D, 2, false>;
    else if (maps != 0u)  // silu / sigmoid (ELU + 1 is for the linear rules only)
      prep = row ? kda_prep_kernel<D, 1, true> : kda_prep_kernel<D, 1, false>;
    else
      prep = row ? kda_prep_kernel<D, 0, true> : kda_prep_kernel<D, 0, false>;
  }
  auto scan = kda_scan_kernel<D, NB, false>;
  if constexpr (D == 128) {
    if (rule == KDA_RULE_LINEAR_NORM) scan = kda_scan_kernel<D, NB, true>;
    else if (nb64) scan = kda_scan_kernel<D, 2 * NB, false>;
  }
  constexpr uint32_t wide_smem = ScanWideSmem::BYTES + 1024;
  const bool pipelined = D == 128 && G > 1 && NC > 0;
  if (cudaFuncSetAttribute(prep, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)prep_smem) != cudaSuccess ||
      cudaFuncSetAttribute(scan, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)scan_smem) != cudaSuccess)
    return KDA_ERR_CUDA;
  if (D == 128 && (wide || pipelined) &&
      cudaFuncSetAttribute(kda_scan_wide_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)wide_smem) != cudaSuccess)
    return KDA_ERR_CUDA;
  const long long total = (long long)BH * NC;
  if (total > 0x7fffffffLL) return KDA_ERR_UNSUPPORTED;
  auto *ob = static_cast<__nv_bfloat16 *>(o);
  auto *qb = static_cast<const __nv_bfloat16 *>(q), *kb = static_cast<const __nv_bfloat16 *>(k),
       *vb = static_cast<const __nv_bfloat16 *>(v);
  const int per_sm = D == 128 ? 2 : 1;  // persistent prep CTAs per SM
  unsigned *claims = D == 128 ? claim_area(ws, BH, NC) : nullptr;
  if (NC > 0 && D == 128 && cudaMemsetAsync(claims, 0, kClaimBytes, st) != cudaSuccess)
    return KDA_ERR_CUDA;
  if (!pipelined) {
    if (NC > 0) {
      const long long slots = (long long)sms * per_sm;
      const int grid = (int)(total < slots ? total : slots);
      timer.mark();
      if (launch_k(prep, dim3(grid), 256, prep_smem, st, false, qb, kb, vb, beta, log_alpha,
                   (int)am, T, NC, (int)total, 0, NC, (int)total, claims, ws, rule, maps,
                   0) != cudaSuccess)
        return KDA_ERR_CUDA;
    }
    timer.mark();
    cudaError_t e;
    if (D == 128 && wide)
      e = launch_k(kda_scan_wide_kernel, dim3(BH), kWideThreads, wide_smem, st, false, h0, ob,
                   hT, T, NC, NC, 0, ws, 0);
    else
      e = launch_k(scan, dim3(D / scan_nbv, BH), D == 128 ? kScan128Threads : kScan64Threads,
                   scan_smem, st, false, h0, ob, hT, T, NC, NC, 0, ws, 0);
    timer.mark();
    return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
  }
  const int seg = (NC + G - 1) / G;
  float *hs = hT ? hT : segment_state(ws, BH, NC);
  // beside a scan segment the prep keeps the SMs the scan leaves free
  const long long side_slots = (long long)(sms > BH ? sms - BH : 1) * per_sm;
  for (int g = 0; g < G; ++g) {
    const int n0 = g * seg;
    const int ns = NC - n0 < seg ? NC - n0 : seg;
    if (ns <= 0) break;
    const bool last = n0 + ns >= NC;
    const long long work = (long long)BH * ns;
    const long long slots = g == 0 ? (long long)sms * per_sm : side_slots;
    timer.mark();
    if (launch_k(prep, dim3((int)(work < slots ? work : slots)), 256, prep_smem, st, g > 0, qb,
                 kb, vb, beta, log_alpha, (int)am, T, NC, (int)total, n0, ns, (int)work,
                 claims + g, ws, rule, maps, 1) != cudaSuccess)
      return KDA_ERR_CUDA;
    const float *hin = g == 0 ? h0 : hs;
    float *hout = last ? hT : hs;
    timer.mark();
    cudaError_t e;
    if (!last)
      e = launch_k(kda_scan_wide_kernel, dim3(BH), kWideThreads, wide_smem, st, true, hin, ob,
                   hout, T, ns, NC, n0, ws, 1);
    else  // the call's last kernel: nothing after it starts early
      e = launch_k(scan, dim3(D / scan_nbv, BH), kScan128Threads, scan_smem, st, true, hin, ob,
                   hout, T, ns, NC, n0, ws, 0);
    if (e != cudaSuccess) return KDA_ERR_CUDA;
  }
  timer.mark();
  return KDA_OK;
}

}  // namespace

bool chunk_tc_supported(int dk, int dv, int C, kda_dtype dt) {
  return dt == KDA_BF16 && C == kC && dk == dv && (dk == 64 || dk == 128);
}

size_t chunk_tc_workspace_bytes(int B, int H, int T, int dk, int dv, int C) {
  if (dk != dv || C != kC) return 0;
  const size_t NC = (size_t)(T + kC - 1) / kC;
  // d = 128: each chunk record is followed, after all of them, by its
  // normaliser sums (read only by the normalised linear-attention rule),
  // those by one state per head (the hand-off between the segments of a
  // pipelined call), and those by the prep's work counters
  if (dk == 128)
    return (size_t)B * H * NC * (Rec<128>::BYTES + NormRec::BYTES) +
           (size_t)B * H * 128 * 128 * sizeof(float) + kClaimBytes;
  return (size_t)B * H * NC * Rec<64>::BYTES;
}

int chunk_tc_segments(int BH, int T, int dk, int rule, int scan) {
  if (dk != 128 || rule == KDA_RULE_LINEAR_NORM || BH <= 0 || T <= 0) return 1;
  const int NC = (T + kC - 1) / kC;
  if (scan == 3) {  // requested: segments of at least 8 chunks, at most 16 of them
    const int g = NC / 8;
    return g < 1 ? 1 : (g > kMaxSegments ? kMaxSegments : g);
  }
  return 1;
}

int chunk_tc_launches(int BH, int T, bool has_hT, int dk, int rule, int scan) {
  if (BH == 0 || (T == 0 && !has_hT)) return 0;
  if (T == 0) return 1;
  const int G = chunk_tc_segments(BH, T, dk, rule, scan);
  if (G == 1) return 2;
  const int NC = (T + kC - 1) / kC, seg = (NC + G - 1) / G;
  return 2 * ((NC + seg - 1) / seg);
}

bool chunk_tc_wide_scan(int BH, int dk, int rule, int scan) {
  if (dk != 128 || rule == KDA_RULE_LINEAR_NORM || scan == 1 || scan == 3) return false;
  if (scan == 2) return true;
  // automatic: the split scan.  The wide scan streams each whole record
  // through one SM; measured on Gated DeltaNet (128 heads, 128 chunks) it
  // took 0.442 ms against 0.434 ms for the split scan in four rounds: there
  // the records' HBM traffic, not the rounds, sets the scan's time.
  return false;
}

const char *chunk_tc_kernel_name(int BH, int T, int dk, int scan, int i) {
  const int n = chunk_tc_launches(BH, T, true, dk, 0, scan);
  if (i < 0 || i >= n) return nullptr;
  if (chunk_tc_segments(BH, T, dk, 0, scan) > 1)  // prep, wide scan, ..., prep, split scan
    return (i & 1) == 0 ? "kda_prep_kernel"
                        : (i == n - 1 ? "kda_scan_kernel" : "kda_scan_wide_kernel");
  const char *scan_name = chunk_tc_wide_scan(BH, dk, 0, scan) ? "kda_scan_wide_kernel"
                                                               : "kda_scan_kernel";
  if (T == 0) return scan_name;
  return i == 0 ? "kda_prep_kernel" : scan_name;
}

kda_status launch_chunk_tc(const void *q, const void *k, const void *v, const float *beta,
                           const float *log_alpha, const float *h0, void *o, float *hT, int B,
                           int H, int T, int dk, int /*dv*/, int /*C*/, kda_alpha_mode am,
                           void *workspace, size_t /*ws_bytes*/, cudaStream_t stream,
                           LaunchTimer &timer, int rule, unsigned maps, int scan) {
  const int BH = B * H;
  if (chunk_tc_launches(BH, T, hT != nullptr, dk, rule, scan) == 0) return KDA_OK;
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  if (dk == 128)
    return launch_d<128>(q, k, v, beta, log_alpha, h0, o, hT, BH, T, am, ws, stream, timer, rule,
                         maps, chunk_tc_wide_scan(BH, dk, rule, scan),
                         chunk_tc_segments(BH, T, dk, rule, scan));
  return launch_d<64>(q, k, v, beta, log_alpha, h0, o, hT, BH, T, am, ws, stream, timer, 0, 0u,
                      false, 1);
}

}  // namespace kda
