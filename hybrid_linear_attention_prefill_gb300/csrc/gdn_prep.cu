// Chunk preparation for the chunked Gated DeltaNet prefill (sm_103a).
//
// For every 64-token chunk and value head this kernel forms the parts of the
// chunk-wise (WY / UT-transform) recurrence that do not depend on the carried
// state.  Within a chunk, with gamma the inclusive cumulative sum of the log
// decays g and Gamma[t][i] = exp(gamma_t - gamma_i) for i <= t:
//
//   A  = strict_lower( diag(beta) (K K^T) * Gamma )      (beta-scaled key Gram)
//   Tm = (I + A)^-1                                      (UT transform, unit lower)
//   P  = lower_incl( (Q K^T) * Gamma )                   (decayed intra-chunk scores)
//   PT = P Tm
//
// Tm and PT are stored as bf16 64 x 64 tiles in the workspace; the state-carry
// kernel combines them with the state.  The pages only name the operation (the
// "chunked Gated DeltaNet prefill" of the "Open-Jev-27B-v1.1 native text
// worker" page, "Validation and optimization scope"); the WY form is the
// standard chunked rewriting of S_t = a_t S_{t-1}(I - b_t k_t k_t^T) + b_t v_t k_t^T.
//
// One CTA handles one chunk slot and one key head, and loops over the value
// heads that share the key head, so the Grams K K^T and Q K^T are computed once
// per key head.  Only non-positive exponents are ever taken (gamma_t - gamma_i,
// i <= t), so nothing overflows however strong the decay.
#include "gdn_common.cuh"

namespace gdn {

template <int DK>
struct PrepSmem {
  static constexpr int LDK = DK + 8;  // bf16 row stride of the K/Q tiles (conflict-free ldmatrix)
  static constexpr int LDF = 68;      // fp32 row stride of 64-wide matrices
  static constexpr int LDB = 72;      // bf16 row stride of 64-wide matrices
  static constexpr int kKQBytes = 2 * kChunk * LDK * 2;
  static constexpr int kATBytes = 2 * kChunk * LDF * 4;
  static constexpr int kUnion = kKQBytes > kATBytes ? kKQBytes : kATBytes;
  // [union: K,Q tiles | A,Tm fp32] [G fp32 x2] [P bf16] [Tm bf16] [W temp] [gamma, beta]
  static constexpr int offG = kUnion;
  static constexpr int offP = offG + 2 * kChunk * LDF * 4;
  static constexpr int offTb = offP + kChunk * LDB * 2;
  static constexpr int offW = offTb + kChunk * LDB * 2;
  static constexpr int offGam = offW + 3 * 16 * 17 * 4;
  static constexpr int bytes = offGam + 2 * kChunk * 4;
};

template <int DK>
__global__ void __launch_bounds__(128)
gdn_prep_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k,
                const float* __restrict__ g, const float* __restrict__ beta,
                const int32_t* __restrict__ cu, const int32_t* __restrict__ chunk_off,
                __nv_bfloat16* __restrict__ ws, int B, int T, int Hk, int Hv, int nc_dense) {
  using L = PrepSmem<DK>;
  extern __shared__ __align__(128) unsigned char smem[];
  __nv_bfloat16* Ks = reinterpret_cast<__nv_bfloat16*>(smem);
  __nv_bfloat16* Qs = Ks + kChunk * L::LDK;
  float* As = reinterpret_cast<float*>(smem);     // aliases K/Q after the Grams
  float* Tms = As + kChunk * L::LDF;
  float* Gs = reinterpret_cast<float*>(smem + L::offG);  // [2][64][LDF]
  __nv_bfloat16* Ps = reinterpret_cast<__nv_bfloat16*>(smem + L::offP);
  __nv_bfloat16* Tmb = reinterpret_cast<__nv_bfloat16*>(smem + L::offTb);
  float* Wt = reinterpret_cast<float*>(smem + L::offW);  // [3][16][17]
  float* gam = reinterpret_cast<float*>(smem + L::offGam);
  float* bet = gam + kChunk;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int slot = blockIdx.x, hk = blockIdx.y;

  // ---- which sequence and chunk this slot is ---------------------------------
  int b, c;
  if (cu == nullptr) {
    b = slot / nc_dense;
    c = slot - b * nc_dense;
    if (b >= B) return;
  } else {
    if (slot >= chunk_off[B]) return;
    int lo = 0, hi = B;  // largest b with chunk_off[b] <= slot
    while (hi - lo > 1) {
      int mid = (lo + hi) >> 1;
      if (chunk_off[mid] <= slot) lo = mid; else hi = mid;
    }
    b = lo;
    c = slot - chunk_off[b];
  }
  const SeqChunk sq = seq_bounds(cu, b, T);
  const long long t0 = sq.bos + (long long)c * kChunk;
  const int n = min(kChunk, sq.len - c * kChunk);

  // ---- load the K and Q tiles (rows >= n are zero) ---------------------------
  {
    constexpr int CPR = DK / 8;  // 16-byte pieces per row
    for (int e = tid; e < kChunk * CPR; e += 128) {
      const int r = e / CPR, p = e - r * CPR;
      const bool ok = r < n;
      const size_t off = ok ? ((size_t)(t0 + r) * Hk + hk) * DK + p * 8 : 0;
      cp_async16(Ks + r * L::LDK + p * 8, k + off, ok);
      cp_async16(Qs + r * L::LDK + p * 8, q + off, ok);
    }
    cp_async_commit();
    cp_async_wait<0>();
    __syncthreads();
  }

  // ---- Grams: G0 = K K^T, G1 = Q K^T on the lower block triangle ------------
  {
    const int mat = warp >> 1;
    const __nv_bfloat16* Asrc = mat == 0 ? Ks : Qs;
    float* Gd = Gs + mat * kChunk * L::LDF;
    const int m = lane >> 3;
#pragma unroll
    for (int s = 0; s < 2; ++s) {
      const int mi = (warp & 1) == 0 ? (s == 0 ? 0 : 3) : (s == 0 ? 1 : 2);
      float acc[8][4];
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
#pragma unroll
      for (int kk = 0; kk < DK / 16; ++kk) {
        uint32_t a[4];
        ldsm_x4(a, Asrc + (16 * mi + 8 * (m & 1) + (lane & 7)) * L::LDK + 16 * kk + 8 * (m >> 1));
#pragma unroll
        for (int p = 0; p < 4; ++p) {
          if (p <= mi) {
            uint32_t bb[4];
            ldsm_x4(bb, Ks + (8 * (2 * p + (m >> 1)) + (lane & 7)) * L::LDK + 16 * kk + 8 * (m & 1));
            mma_bf16(acc[2 * p], a, bb[0], bb[1]);
            mma_bf16(acc[2 * p + 1], a, bb[2], bb[3]);
          }
        }
      }
      const int r0 = 16 * mi + (lane >> 2);
#pragma unroll
      for (int nj = 0; nj < 8; ++nj) {
        if (nj <= 2 * mi + 1) {
          const int cc = 8 * nj + 2 * (lane & 3);
          *reinterpret_cast<float2*>(Gd + r0 * L::LDF + cc) = make_float2(acc[nj][0], acc[nj][1]);
          *reinterpret_cast<float2*>(Gd + (r0 + 8) * L::LDF + cc) = make_float2(acc[nj][2], acc[nj][3]);
        }
      }
    }
  }
  __syncthreads();

  const int G = Hv / Hk;
  for (int gi = 0; gi < G; ++gi) {
    const int h = hk * G + gi;
    // ---- gamma = inclusive cumsum of g in the chunk -------------------------
    if (warp == 0) {
      float g0 = 0.f, g1 = 0.f, b0 = 0.f, b1 = 0.f;
      if (lane < n) { g0 = g[(t0 + lane) * Hv + h]; b0 = beta[(t0 + lane) * Hv + h]; }
      if (lane + 32 < n) { g1 = g[(t0 + lane + 32) * Hv + h]; b1 = beta[(t0 + lane + 32) * Hv + h]; }
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float u0 = __shfl_up_sync(0xffffffffu, g0, o);
        const float u1 = __shfl_up_sync(0xffffffffu, g1, o);
        if (lane >= o) { g0 += u0; g1 += u1; }
      }
      g1 += __shfl_sync(0xffffffffu, g0, 31);
      gam[lane] = g0;
      gam[lane + 32] = g1;
      bet[lane] = b0;
      bet[lane + 32] = b1;
    }
    __syncthreads();

    // ---- A (fp32) and P (bf16) -------------------------------------------------
    for (int e = tid; e < kChunk * kChunk; e += 128) {
      const int t = e >> 6, i = e & 63;
      float a = 0.f, p = 0.f;
      if (i <= t) {
        const float d = expf(gam[t] - gam[i]);
        p = d * Gs[kChunk * L::LDF + t * L::LDF + i];
        if (i < t) a = bet[t] * d * Gs[t * L::LDF + i];
      }
      As[t * L::LDF + i] = a;
      Ps[t * L::LDB + i] = __float2bfloat16_rn(p);
    }
    // zero the strictly-upper 16x16 blocks of Tm
    for (int e = tid; e < 6 * 256; e += 128) {
      const int blk = e >> 8, w = e & 255;
      const int bi = blk < 3 ? 0 : (blk < 5 ? 1 : 2);
      const int bj = blk < 3 ? blk + 1 : (blk < 5 ? blk - 1 : 3);
      Tms[(16 * bi + (w >> 4)) * L::LDF + 16 * bj + (w & 15)] = 0.f;
    }
    __syncthreads();

    // ---- Tm = (I + A)^-1: diagonal 16x16 blocks by forward substitution ------
    if (tid < 64) {
      const int blk = tid >> 4, j = tid & 15;
      const float* Ab = As + 16 * blk * L::LDF + 16 * blk;
      float x[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) x[i] = (i == j) ? 1.f : 0.f;
#pragma unroll
      for (int t = 1; t < 16; ++t) {
        float s = 0.f;
#pragma unroll
        for (int i = 0; i < t; ++i) s = fmaf(Ab[t * L::LDF + i], x[i], s);
        if (t > j) x[t] = -s;
      }
      float* Tb = Tms + 16 * blk * L::LDF + 16 * blk;
#pragma unroll
      for (int t = 0; t < 16; ++t) Tb[t * L::LDF + j] = x[t];
    }
    __syncthreads();
    // ---- off-diagonal blocks, one block row at a time ------------------------
    //   Tm_ij = -Tm_ii * sum_{kb=j}^{i-1} A_{i,kb} Tm_{kb,j}
    for (int bi = 1; bi < 4; ++bi) {
      for (int e = tid; e < bi * 256; e += 128) {
        const int bj = e >> 8, r = (e >> 4) & 15, cc = e & 15;
        const float* Ar = As + (16 * bi + r) * L::LDF;
        float s = 0.f;
        for (int kb = bj; kb < bi; ++kb) {
#pragma unroll
          for (int mm = 0; mm < 16; ++mm)
            s = fmaf(Ar[16 * kb + mm], Tms[(16 * kb + mm) * L::LDF + 16 * bj + cc], s);
        }
        Wt[(bj * 16 + r) * 17 + cc] = s;
      }
      __syncthreads();
      for (int e = tid; e < bi * 256; e += 128) {
        const int bj = e >> 8, r = (e >> 4) & 15, cc = e & 15;
        const float* Tr = Tms + (16 * bi + r) * L::LDF + 16 * bi;
        float s = 0.f;
#pragma unroll
        for (int mm = 0; mm < 16; ++mm)
          if (mm <= r) s = fmaf(Tr[mm], Wt[(bj * 16 + mm) * 17 + cc], s);
        Tms[(16 * bi + r) * L::LDF + 16 * bj + cc] = -s;
      }
      __syncthreads();
    }

    // ---- bf16 Tm: to shared (for PT) and to the workspace ---------------------
    __nv_bfloat16* wsT = ws + ((size_t)slot * Hv + h) * (2 * kWsTileElems);
    __nv_bfloat16* wsPT = wsT + kWsTileElems;
    for (int e = tid; e < kChunk * 8; e += 128) {
      const int r = e >> 3, p = e & 7;
      const float* src = Tms + r * L::LDF + 8 * p;
      uint4 v;
      v.x = pack_bf16(src[0], src[1]);
      v.y = pack_bf16(src[2], src[3]);
      v.z = pack_bf16(src[4], src[5]);
      v.w = pack_bf16(src[6], src[7]);
      *reinterpret_cast<uint4*>(Tmb + r * L::LDB + 8 * p) = v;
      *reinterpret_cast<uint4*>(wsT + r * kChunk + 8 * p) = v;
    }
    __syncthreads();

    // ---- PT = P Tm (lower triangular); warp w owns rows 16w..16w+15 ----------
    {
      const int m = lane >> 3;
      float acc[8][4];
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        if (kk <= warp) {
          uint32_t a[4];
          ldsm_x4(a, Ps + (16 * warp + 8 * (m & 1) + (lane & 7)) * L::LDB + 16 * kk + 8 * (m >> 1));
#pragma unroll
          for (int p = 0; p < 4; ++p) {
            if (p <= kk) {  // columns j < 16(kk+1) only
              uint32_t bb[4];
              ldsm_x4_t(bb, Tmb + (16 * kk + 8 * (m & 1) + (lane & 7)) * L::LDB + 8 * (2 * p + (m >> 1)));
              mma_bf16(acc[2 * p], a, bb[0], bb[1]);
              mma_bf16(acc[2 * p + 1], a, bb[2], bb[3]);
            }
          }
        }
      }
      __syncwarp();
      // each warp overwrites only its own rows of Ps, which only it reads
      const int r0 = 16 * warp + (lane >> 2);
#pragma unroll
      for (int nj = 0; nj < 8; ++nj) {
        const int cc = 8 * nj + 2 * (lane & 3);
        *reinterpret_cast<uint32_t*>(Ps + r0 * L::LDB + cc) = pack_bf16(acc[nj][0], acc[nj][1]);
        *reinterpret_cast<uint32_t*>(Ps + (r0 + 8) * L::LDB + cc) = pack_bf16(acc[nj][2], acc[nj][3]);
      }
    }
    __syncthreads();
    for (int e = tid; e < kChunk * 8; e += 128) {
      const int r = e >> 3, p = e & 7;
      *reinterpret_cast<uint4*>(wsPT + r * kChunk + 8 * p) =
          *reinterpret_cast<const uint4*>(Ps + r * L::LDB + 8 * p);
    }
    __syncthreads();
  }
}

// Prefix sums of chunk counts for packed sequences: chunk_off[b] = sum over
// b' < b of ceil(len_b' / 64), chunk_off[B] = total.  One CTA of 1024 threads.
__global__ void __launch_bounds__(1024)
gdn_chunk_table_kernel(const int32_t* __restrict__ cu, int B, int T, int32_t* __restrict__ chunk_off) {
  __shared__ int wsum[32];
  __shared__ int carry;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) carry = 0;
  __syncthreads();
  for (int base = 0; base < B; base += 1024) {
    const int b = base + tid;
    int nc = 0;
    if (b < B) {
      const SeqChunk s = seq_bounds(cu, b, T);
      nc = (s.len + kChunk - 1) / kChunk;
    }
    int x = nc;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) wsum[warp] = x;
    __syncthreads();
    if (warp == 0) {
      int w = wsum[lane];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, w, o);
        if (lane >= o) w += y;
      }
      wsum[lane] = w;  // inclusive over warps
    }
    __syncthreads();
    const int excl = carry + (warp ? wsum[warp - 1] : 0) + x - nc;
    if (b < B) chunk_off[b] = excl;
    __syncthreads();
    if (tid == 0) carry += wsum[31];
    __syncthreads();
  }
  if (tid == 0) chunk_off[B] = carry;
}

// ---- launchers -----------------------------------------------------------------
template <int DK>
cudaError_t launch_prep(const void* q, const void* k, const float* g, const float* beta,
                        const int32_t* cu, const int32_t* chunk_off, void* ws, int B, int T,
                        int Hk, int Hv, int nslots, int nc_dense, cudaStream_t st) {
  using L = PrepSmem<DK>;
  cudaError_t e = cudaFuncSetAttribute(gdn_prep_kernel<DK>, cudaFuncAttributeMaxDynamicSharedMemorySize, L::bytes);
  if (e != cudaSuccess) return e;
  dim3 grid(nslots, Hk);
  gdn_prep_kernel<DK><<<grid, 128, L::bytes, st>>>(
      static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(k), g, beta, cu, chunk_off,
      static_cast<__nv_bfloat16*>(ws), B, T, Hk, Hv, nc_dense);
  return cudaGetLastError();
}

cudaError_t launch_chunk_table(const int32_t* cu, int B, int T, int32_t* chunk_off, cudaStream_t st) {
  gdn_chunk_table_kernel<<<1, 1024, 0, st>>>(cu, B, T, chunk_off);
  return cudaGetLastError();
}

template cudaError_t launch_prep<32>(const void*, const void*, const float*, const float*, const int32_t*,
                                     const int32_t*, void*, int, int, int, int, int, int, cudaStream_t);
template cudaError_t launch_prep<64>(const void*, const void*, const float*, const float*, const int32_t*,
                                     const int32_t*, void*, int, int, int, int, int, int, cudaStream_t);
template cudaError_t launch_prep<128>(const void*, const void*, const float*, const float*, const int32_t*,
                                      const int32_t*, void*, int, int, int, int, int, int, cudaStream_t);

}  // namespace gdn
