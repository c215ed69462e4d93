// Chunk-sequential state carry for the chunked Gated DeltaNet prefill (sm_103a).
//
// Per (sequence, value head, 32-row slice of the dv x dk state S) one CTA walks
// the sequence's 64-token chunks in order.  For a chunk that starts from S
// (n tokens; rows beyond n are zero, with g = beta = 0), using the workspace
// tiles Tm = (I + A)^-1 and PT = P Tm written by the preparation kernel and
// gamma = cumsum(g), e = exp(gamma), d = exp(gamma_last - gamma):
//
//   R   = diag(beta) V - diag(beta e) K S^T          (new values minus what S predicts)
//   U   = Tm R                                       (the delta-rule corrections u_t)
//   O   = scale (diag(e) Q S^T + PT R)               (outputs, scale = 1/sqrt(dk))
//   S  <- e_last S + U^T diag(d) K                   (state after the chunk)
//
// This is the chunk form of S_t = a_t S_{t-1}(I - b_t k_t k_t^T) + b_t v_t k_t^T,
// o_t = S_t q_t / sqrt(dk) ("chunked Gated DeltaNet prefill", "Open-Jev-27B-v1.1
// native text worker", section "Validation and optimization scope"); rows of S
// evolve independently, so slicing dv is exact.
//
// Each warp owns 16 rows of S in fp32 registers for the whole sequence and
// computes every product of its chain with mma.sync bf16 tensor-core tiles,
// transposed so the state is the M dimension:  X^T = S K^T, Y^T = S Q^T,
// [U | PT R]^T = R^T [Tm | PT]^T, dS = (diag(d) U)^T K.  Operands that carry
// the state (S in S K^T, R, and diag(d) U) are split into bf16 hi + lo parts so
// the fp32 state keeps ~2^-16 relative accuracy; output-only products use the
// hi parts.
#include "gdn_common.cuh"

namespace gdn {

template <int DK, int DVT>
struct ChainSmem {
  static constexpr int LDK = DK + 8;
  static constexpr int LDV = DVT + 8;
  static constexpr int LDT = kChunk + 8;
  // one stage: K, Q, V, Tm, PT (bf16), g, beta (fp32)
  static constexpr int offQ = kChunk * LDK * 2;
  static constexpr int offV = offQ + kChunk * LDK * 2;
  static constexpr int offT = offV + kChunk * LDV * 2;
  static constexpr int offPT = offT + kChunk * LDT * 2;
  static constexpr int offG = offPT + kChunk * LDT * 2;
  static constexpr int offB = offG + kChunk * 4;
  static constexpr int stage = offB + kChunk * 4;
  // after the two stages: output staging and per-token scalars
  static constexpr int offO = 2 * stage;
  static constexpr int offS = offO + kChunk * LDV * 2;
  static constexpr int bytes = offS + (4 * kChunk + 4) * 4;
};

template <int DK, int DVT>
__global__ void __launch_bounds__(DVT * 2)
gdn_chain_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k,
                 const __nv_bfloat16* __restrict__ v, const float* __restrict__ g,
                 const float* __restrict__ beta, const int32_t* __restrict__ cu,
                 const int32_t* __restrict__ chunk_off, const __nv_bfloat16* __restrict__ ws,
                 const float* init, __nv_bfloat16* __restrict__ out, float* fin,
                 int B, int T, int Hk, int Hv, int DV, int nc_dense, long long nslots) {
  using L = ChainSmem<DK, DVT>;
  constexpr int NT = DVT * 2;  // threads: one warp per 16 rows
  extern __shared__ __align__(128) unsigned char smem[];
  float* s_b = reinterpret_cast<float*>(smem + L::offS);  // beta
  float* s_be = s_b + kChunk;                             // beta * e
  float* s_es = s_be + kChunk;                            // scale * e
  float* s_d = s_es + kChunk;                             // exp(gamma_last - gamma)
  float* s_eC = s_d + kChunk;                             // exp(gamma_last)
  __nv_bfloat16* Os = reinterpret_cast<__nv_bfloat16*>(smem + L::offO);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int ntiles = DV / DVT;
  const int b = blockIdx.x / ntiles;
  const int dv0 = (blockIdx.x - b * ntiles) * DVT;
  const int h = blockIdx.y;
  const int hk = h / (Hv / Hk);
  const float scale = rsqrtf((float)DK);

  const SeqChunk sq = seq_bounds(cu, b, T);
  const int slot0 = cu == nullptr ? b * nc_dense : chunk_off[b];
  // chunks of this sequence; never past the workspace, even for malformed cu_seqlens
  int nchunks = (sq.len + kChunk - 1) / kChunk;
  if ((long long)slot0 + nchunks > nslots) nchunks = slot0 < nslots ? (int)(nslots - slot0) : 0;

  // ---- initial state: rows dv0 + 16 warp + {g8, g8 + 8}, fp32 accumulator layout
  const int g8 = lane >> 2, tig = lane & 3;
  float S[DK / 8][4];
  {
    const size_t base = ((size_t)b * Hv + h) * DV + dv0 + 16 * warp;
#pragma unroll
    for (int nt = 0; nt < DK / 8; ++nt) {
      float2 lo = make_float2(0.f, 0.f), hi = make_float2(0.f, 0.f);
      if (init != nullptr) {
        lo = *reinterpret_cast<const float2*>(init + (base + g8) * DK + 8 * nt + 2 * tig);
        hi = *reinterpret_cast<const float2*>(init + (base + g8 + 8) * DK + 8 * nt + 2 * tig);
      }
      S[nt][0] = lo.x; S[nt][1] = lo.y; S[nt][2] = hi.x; S[nt][3] = hi.y;
    }
  }

  auto load_chunk = [&](int c, int stg) {
    unsigned char* st = smem + stg * L::stage;
    __nv_bfloat16* Ks = reinterpret_cast<__nv_bfloat16*>(st);
    __nv_bfloat16* Qs = reinterpret_cast<__nv_bfloat16*>(st + L::offQ);
    __nv_bfloat16* Vs = reinterpret_cast<__nv_bfloat16*>(st + L::offV);
    __nv_bfloat16* Ts = reinterpret_cast<__nv_bfloat16*>(st + L::offT);
    __nv_bfloat16* PTs = reinterpret_cast<__nv_bfloat16*>(st + L::offPT);
    float* gs = reinterpret_cast<float*>(st + L::offG);
    float* bs = reinterpret_cast<float*>(st + L::offB);
    const long long t0 = sq.bos + (long long)c * kChunk;
    const int n = min(kChunk, sq.len - c * kChunk);
    constexpr int CPK = DK / 8;
    for (int e = tid; e < kChunk * CPK; e += NT) {
      const int r = e / CPK, p = e - r * CPK;
      const bool ok = r < n;
      const size_t off = ok ? ((size_t)(t0 + r) * Hk + hk) * DK + p * 8 : 0;
      cp_async16(Ks + r * L::LDK + p * 8, k + off, ok);
      cp_async16(Qs + r * L::LDK + p * 8, q + off, ok);
    }
    constexpr int CPV = DVT / 8;
    for (int e = tid; e < kChunk * CPV; e += NT) {
      const int r = e / CPV, p = e - r * CPV;
      const bool ok = r < n;
      const size_t off = ok ? ((size_t)(t0 + r) * Hv + h) * DV + dv0 + p * 8 : 0;
      cp_async16(Vs + r * L::LDV + p * 8, v + off, ok);
    }
    const __nv_bfloat16* wt = ws + ((size_t)(slot0 + c) * Hv + h) * (2 * kWsTileElems);
    for (int e = tid; e < kChunk * 8; e += NT) {
      const int r = e >> 3, p = e & 7;
      cp_async16(Ts + r * L::LDT + p * 8, wt + r * kChunk + p * 8, true);
      cp_async16(PTs + r * L::LDT + p * 8, wt + kWsTileElems + r * kChunk + p * 8, true);
    }
    for (int r = tid; r < kChunk; r += NT) {
      const bool ok = r < n;
      const size_t off = ok ? (size_t)(t0 + r) * Hv + h : 0;
      cp_async4(gs + r, g + off, ok);
      cp_async4(bs + r, beta + off, ok);
    }
  };

  if (nchunks > 0) load_chunk(0, 0);
  cp_async_commit();

  const int m = lane >> 3;
  const int rw = 16 * warp;  // this warp's first row within the slice

  for (int c = 0; c < nchunks; ++c) {
    const int stg = c & 1;
    if (c + 1 < nchunks) load_chunk(c + 1, stg ^ 1);
    cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();

    unsigned char* st = smem + stg * L::stage;
    const __nv_bfloat16* Ks = reinterpret_cast<const __nv_bfloat16*>(st);
    const __nv_bfloat16* Qs = reinterpret_cast<const __nv_bfloat16*>(st + L::offQ);
    const __nv_bfloat16* Vs = reinterpret_cast<const __nv_bfloat16*>(st + L::offV);
    const __nv_bfloat16* Ts = reinterpret_cast<const __nv_bfloat16*>(st + L::offT);
    const __nv_bfloat16* PTs = reinterpret_cast<const __nv_bfloat16*>(st + L::offPT);
    const float* gs = reinterpret_cast<const float*>(st + L::offG);
    const float* bs = reinterpret_cast<const float*>(st + L::offB);

    // ---- per-token scalars (warp 0) ---------------------------------------------
    if (warp == 0) {
      float g0 = gs[lane], g1 = gs[lane + 32];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float u0 = __shfl_up_sync(0xffffffffu, g0, o);
        const float u1 = __shfl_up_sync(0xffffffffu, g1, o);
        if (lane >= o) { g0 += u0; g1 += u1; }
      }
      g1 += __shfl_sync(0xffffffffu, g0, 31);
      const float gl = __shfl_sync(0xffffffffu, g1, 31);
      const float e0 = expf(g0), e1 = expf(g1);
      const float b0 = bs[lane], b1 = bs[lane + 32];
      s_b[lane] = b0; s_b[lane + 32] = b1;
      s_be[lane] = b0 * e0; s_be[lane + 32] = b1 * e1;
      s_es[lane] = scale * e0; s_es[lane + 32] = scale * e1;
      s_d[lane] = expf(gl - g0); s_d[lane + 32] = expf(gl - g1);
      if (lane == 0) s_eC[0] = expf(gl);
    }
    __syncthreads();

    // ---- X^T = S K^T (hi + lo), Y^T = S Q^T (hi) ---------------------------------
    float X[8][4], Y[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) X[i][j] = Y[i][j] = 0.f;
#pragma unroll
    for (int kk = 0; kk < DK / 16; ++kk) {
      uint32_t ah[4], al[4];
      split_bf16(S[2 * kk][0], S[2 * kk][1], ah[0], al[0]);
      split_bf16(S[2 * kk][2], S[2 * kk][3], ah[1], al[1]);
      split_bf16(S[2 * kk + 1][0], S[2 * kk + 1][1], ah[2], al[2]);
      split_bf16(S[2 * kk + 1][2], S[2 * kk + 1][3], ah[3], al[3]);
#pragma unroll
      for (int p = 0; p < 4; ++p) {
        const int row = 8 * (2 * p + (m >> 1)) + (lane & 7);
        const int col = 16 * kk + 8 * (m & 1);
        uint32_t bk[4], bq[4];
        ldsm_x4(bk, Ks + row * L::LDK + col);
        ldsm_x4(bq, Qs + row * L::LDK + col);
        mma_bf16(X[2 * p], ah, bk[0], bk[1]);
        mma_bf16(X[2 * p], al, bk[0], bk[1]);
        mma_bf16(X[2 * p + 1], ah, bk[2], bk[3]);
        mma_bf16(X[2 * p + 1], al, bk[2], bk[3]);
        mma_bf16(Y[2 * p], ah, bq[0], bq[1]);
        mma_bf16(Y[2 * p + 1], ah, bq[2], bq[3]);
      }
    }

    // ---- R^T = diag(beta) V^T - (S K^T) diag(beta e), split into A fragments ----
    uint32_t rh[4][4], rl[4][4];
#pragma unroll
    for (int tn = 0; tn < 8; ++tn) {
      float r4[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int t = 8 * tn + 2 * tig + (e & 1);
        const int r = g8 + 8 * (e >> 1);
        r4[e] = s_b[t] * __bfloat162float(Vs[t * L::LDV + rw + r]) - s_be[t] * X[tn][e];
      }
      const int kk2 = tn >> 1, hlf = tn & 1;
      split_bf16(r4[0], r4[1], rh[kk2][2 * hlf], rl[kk2][2 * hlf]);
      split_bf16(r4[2], r4[3], rh[kk2][2 * hlf + 1], rl[kk2][2 * hlf + 1]);
    }

    // ---- U^T = R^T Tm^T and (PT R)^T = R^T PT^T (both lower triangular) -----------
    float U[8][4], OP[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) U[i][j] = OP[i][j] = 0.f;
#pragma unroll
    for (int kk2 = 0; kk2 < 4; ++kk2) {
#pragma unroll
      for (int p = 0; p < 4; ++p) {
        if (kk2 <= p) {
          const int row = 8 * (2 * p + (m >> 1)) + (lane & 7);
          const int col = 16 * kk2 + 8 * (m & 1);
          uint32_t bt[4], bp[4];
          ldsm_x4(bt, Ts + row * L::LDT + col);
          ldsm_x4(bp, PTs + row * L::LDT + col);
          mma_bf16(U[2 * p], rh[kk2], bt[0], bt[1]);
          mma_bf16(U[2 * p], rl[kk2], bt[0], bt[1]);
          mma_bf16(U[2 * p + 1], rh[kk2], bt[2], bt[3]);
          mma_bf16(U[2 * p + 1], rl[kk2], bt[2], bt[3]);
          mma_bf16(OP[2 * p], rh[kk2], bp[0], bp[1]);
          mma_bf16(OP[2 * p], rl[kk2], bp[0], bp[1]);
          mma_bf16(OP[2 * p + 1], rh[kk2], bp[2], bp[3]);
          mma_bf16(OP[2 * p + 1], rl[kk2], bp[2], bp[3]);
        }
      }
    }

    // ---- outputs to the staging tile; U^T diag(d) as split A fragments ----------
    uint32_t uh[4][4], ul[4][4];
#pragma unroll
    for (int tn = 0; tn < 8; ++tn) {
      float u4[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int t = 8 * tn + 2 * tig + (e & 1);
        const int r = g8 + 8 * (e >> 1);
        const float o = s_es[t] * Y[tn][e] + scale * OP[tn][e];
        Os[t * L::LDV + rw + r] = __float2bfloat16_rn(o);
        u4[e] = s_d[t] * U[tn][e];
      }
      const int kk2 = tn >> 1, hlf = tn & 1;
      split_bf16(u4[0], u4[1], uh[kk2][2 * hlf], ul[kk2][2 * hlf]);
      split_bf16(u4[2], u4[3], uh[kk2][2 * hlf + 1], ul[kk2][2 * hlf + 1]);
    }

    // ---- S <- e_last S + (diag(d) U)^T K ------------------------------------------
    const float eC = s_eC[0];
#pragma unroll
    for (int nt = 0; nt < DK / 8; ++nt)
#pragma unroll
      for (int j = 0; j < 4; ++j) S[nt][j] *= eC;
#pragma unroll
    for (int kk2 = 0; kk2 < 4; ++kk2) {
#pragma unroll
      for (int np = 0; np < DK / 16; ++np) {
        uint32_t bk[4];
        ldsm_x4_t(bk, Ks + (16 * kk2 + 8 * (m & 1) + (lane & 7)) * L::LDK + 8 * (2 * np + (m >> 1)));
        mma_bf16(S[2 * np], uh[kk2], bk[0], bk[1]);
        mma_bf16(S[2 * np], ul[kk2], bk[0], bk[1]);
        mma_bf16(S[2 * np + 1], uh[kk2], bk[2], bk[3]);
        mma_bf16(S[2 * np + 1], ul[kk2], bk[2], bk[3]);
      }
    }
    __syncthreads();

    // ---- staged outputs to HBM (16-byte pieces, rows < n) ------------------------
    {
      const long long t0 = sq.bos + (long long)c * kChunk;
      const int n = min(kChunk, sq.len - c * kChunk);
      constexpr int CPV = DVT / 8;
      for (int e = tid; e < n * CPV; e += NT) {
        const int r = e / CPV, p = e - r * CPV;
        *reinterpret_cast<uint4*>(out + ((size_t)(t0 + r) * Hv + h) * DV + dv0 + p * 8) =
            *reinterpret_cast<const uint4*>(Os + r * L::LDV + p * 8);
      }
    }
    // the next iteration's first barrier orders these reads before Os is rewritten
  }

  // ---- final state -------------------------------------------------------------------
  if (fin != nullptr) {
    const size_t base = ((size_t)b * Hv + h) * DV + dv0 + 16 * warp;
#pragma unroll
    for (int nt = 0; nt < DK / 8; ++nt) {
      *reinterpret_cast<float2*>(fin + (base + g8) * DK + 8 * nt + 2 * tig) = make_float2(S[nt][0], S[nt][1]);
      *reinterpret_cast<float2*>(fin + (base + g8 + 8) * DK + 8 * nt + 2 * tig) = make_float2(S[nt][2], S[nt][3]);
    }
  }
}

template <int DK>
cudaError_t launch_chain(const void* q, const void* k, const void* v, const float* g, const float* beta,
                         const int32_t* cu, const int32_t* chunk_off, const void* ws, const float* init,
                         void* out, float* fin, int B, int T, int Hk, int Hv, int DV, int nc_dense,
                         long long nslots, cudaStream_t st) {
  constexpr int DVT = 32;
  using L = ChainSmem<DK, DVT>;
  cudaError_t e = cudaFuncSetAttribute(gdn_chain_kernel<DK, DVT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       L::bytes);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)B * (DV / DVT), Hv);
  gdn_chain_kernel<DK, DVT><<<grid, DVT * 2, L::bytes, st>>>(
      static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(k),
      static_cast<const __nv_bfloat16*>(v), g, beta, cu, chunk_off, static_cast<const __nv_bfloat16*>(ws), init,
      static_cast<__nv_bfloat16*>(out), fin, B, T, Hk, Hv, DV, nc_dense, nslots);
  return cudaGetLastError();
}

#define GDN_INST_CHAIN(DK)                                                                                 \
  template cudaError_t launch_chain<DK>(const void*, const void*, const void*, const float*, const float*, \
                                        const int32_t*, const int32_t*, const void*, const float*, void*,  \
                                        float*, int, int, int, int, int, int, long long, cudaStream_t);
GDN_INST_CHAIN(32)
GDN_INST_CHAIN(64)
GDN_INST_CHAIN(128)

}  // namespace gdn
