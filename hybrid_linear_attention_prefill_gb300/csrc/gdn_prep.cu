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
// One CTA (8 warps) handles one chunk slot and one key head, and loops over the
// value heads that share the key head, so the Grams K K^T and Q K^T are computed
// once per key head.  The inverse is blocked: the four 16 x 16 diagonal blocks
// by forward substitution in fp32, then the 16 -> 32 -> 64 merges
// T21 = -T22 A21 T11 as tensor-core products whose fp32 operands are split into
// bf16 hi + lo parts (hi*hi + hi*lo + lo*hi, ~2^-16 relative).  Only non-positive
// exponents are ever taken (gamma_t - gamma_i, i <= t), so nothing overflows
// however strong the decay.
#include "gdn_common.cuh"

namespace gdn {

namespace {

constexpr int kPrepThreads = 256;
constexpr int LDF = 68;  // fp32 row stride of 64-wide matrices
constexpr int LDB = 72;  // bf16 row stride of 64-wide matrices
constexpr int LDW = 36;  // fp32 row stride of the 32-wide merge buffer

// acc (16 x 8 tile) += X[r0:r0+16, k0:k0+16] * Y[ky:ky+16, n0:n0+8] for fp32 X, Y in
// shared memory, as three bf16 products of the hi / lo splits.
__device__ __forceinline__ void mma_f32x3(float (&acc)[4], const float* X, int ldx, int r0, int k0,
                                          const float* Y, int ldy, int ky, int n0, int lane) {
  const int g8 = lane >> 2, tg = lane & 3;
  const float2 x0 = *reinterpret_cast<const float2*>(X + (r0 + g8) * ldx + k0 + 2 * tg);
  const float2 x1 = *reinterpret_cast<const float2*>(X + (r0 + g8 + 8) * ldx + k0 + 2 * tg);
  const float2 x2 = *reinterpret_cast<const float2*>(X + (r0 + g8) * ldx + k0 + 8 + 2 * tg);
  const float2 x3 = *reinterpret_cast<const float2*>(X + (r0 + g8 + 8) * ldx + k0 + 8 + 2 * tg);
  uint32_t ah[4], al[4];
  split_bf16(x0.x, x0.y, ah[0], al[0]);
  split_bf16(x1.x, x1.y, ah[1], al[1]);
  split_bf16(x2.x, x2.y, ah[2], al[2]);
  split_bf16(x3.x, x3.y, ah[3], al[3]);
  uint32_t bh0, bl0, bh1, bl1;
  split_bf16(Y[(ky + 2 * tg) * ldy + n0 + g8], Y[(ky + 2 * tg + 1) * ldy + n0 + g8], bh0, bl0);
  split_bf16(Y[(ky + 2 * tg + 8) * ldy + n0 + g8], Y[(ky + 2 * tg + 9) * ldy + n0 + g8], bh1, bl1);
  mma_bf16(acc, ah, bh0, bh1);
  mma_bf16(acc, ah, bl0, bl1);
  mma_bf16(acc, al, bh0, bh1);
}

// Store a 16 x 8 accumulator tile (times `sgn`) at D[r0.., n0..].
__device__ __forceinline__ void store_tile(float* D, int ldd, int r0, int n0, const float (&acc)[4], float sgn,
                                           int lane) {
  const int g8 = lane >> 2, tg = lane & 3;
  *reinterpret_cast<float2*>(D + (r0 + g8) * ldd + n0 + 2 * tg) = make_float2(sgn * acc[0], sgn * acc[1]);
  *reinterpret_cast<float2*>(D + (r0 + g8 + 8) * ldd + n0 + 2 * tg) = make_float2(sgn * acc[2], sgn * acc[3]);
}

}  // namespace

template <int DK>
struct PrepSmem {
  static constexpr int LDK = DK + 8;  // bf16 row stride of the K/Q tiles (conflict-free ldmatrix)
  static constexpr int kKQBytes = 2 * kChunk * LDK * 2;
  static constexpr int kATBytes = 2 * kChunk * LDF * 4;
  static constexpr int kUnion = kKQBytes > kATBytes ? kKQBytes : kATBytes;
  // [union: K,Q tiles | A,Tm fp32] [G fp32 x2] [P bf16] [Tm bf16] [merge buffer] [gamma, beta]
  static constexpr int offG = kUnion;
  static constexpr int offP = offG + 2 * kChunk * LDF * 4;
  static constexpr int offTb = offP + kChunk * LDB * 2;
  static constexpr int offW = offTb + kChunk * LDB * 2;
  static constexpr int offGam = offW + 32 * LDW * 4;
  static constexpr int bytes = offGam + 2 * kChunk * 4;
};

template <int DK>
__global__ void __launch_bounds__(kPrepThreads, 2)
gdn_prep_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k,
                const float* __restrict__ g, const float* __restrict__ beta,
                const int32_t* __restrict__ cu, const int32_t* __restrict__ chunk_off,
                __nv_bfloat16* __restrict__ ws, int B, int T, int Hk, int Hv, int nc_dense) {
  using L = PrepSmem<DK>;
  extern __shared__ __align__(128) unsigned char smem[];
  __nv_bfloat16* Ks = reinterpret_cast<__nv_bfloat16*>(smem);
  __nv_bfloat16* Qs = Ks + kChunk * L::LDK;
  float* As = reinterpret_cast<float*>(smem);  // aliases K/Q after the Grams
  float* Tms = As + kChunk * LDF;
  float* Gs = reinterpret_cast<float*>(smem + L::offG);  // [2][64][LDF]
  __nv_bfloat16* Ps = reinterpret_cast<__nv_bfloat16*>(smem + L::offP);
  __nv_bfloat16* Tmb = reinterpret_cast<__nv_bfloat16*>(smem + L::offTb);
  float* Wt = reinterpret_cast<float*>(smem + L::offW);  // [32][LDW]
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
      const int mid = (lo + hi) >> 1;
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
    for (int e = tid; e < kChunk * CPR; e += kPrepThreads) {
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
    const int mat = warp >> 2, mi = warp & 3;
    const __nv_bfloat16* Asrc = mat == 0 ? Ks : Qs;
    float* Gd = Gs + mat * kChunk * LDF;
    const int m = lane >> 3;
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
#pragma unroll
    for (int nj = 0; nj < 8; ++nj)
      if (nj <= 2 * mi + 1) store_tile(Gd, LDF, 16 * mi, 8 * nj, acc[nj], 1.f, lane);
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

    // ---- A (fp32), P (bf16); zero the blocks of Tm above the diagonal --------
    for (int e = tid; e < kChunk * kChunk; e += kPrepThreads) {
      const int t = e >> 6, i = e & 63;
      float a = 0.f, p = 0.f;
      if (i <= t) {
        const float dcy = expf(gam[t] - gam[i]);
        p = dcy * Gs[kChunk * LDF + t * LDF + i];
        if (i < t) a = bet[t] * dcy * Gs[t * LDF + i];
      }
      As[t * LDF + i] = a;
      Ps[t * LDB + i] = __float2bfloat16_rn(p);
      if ((i >> 4) > (t >> 4)) Tms[t * LDF + i] = 0.f;
    }
    __syncthreads();

    // ---- Tm: the four 16 x 16 diagonal blocks by forward substitution --------
    if (tid < 64) {
      const int blk = tid >> 4, j = tid & 15;
      const float* Ab = As + 16 * blk * LDF + 16 * blk;
      float x[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) x[i] = (i == j) ? 1.f : 0.f;
#pragma unroll
      for (int t = 1; t < 16; ++t) {
        float s = 0.f;
#pragma unroll
        for (int i = 0; i < t; ++i) s = fmaf(Ab[t * LDF + i], x[i], s);
        if (t > j) x[t] = -s;
      }
      float* Tb = Tms + 16 * blk * LDF + 16 * blk;
#pragma unroll
      for (int t = 0; t < 16; ++t) Tb[t * LDF + j] = x[t];
    }
    __syncthreads();

    // ---- merge 16 -> 32: T[o+16.., o..] = -T22 (A21 T11), o = 0 and 32 -------
    if (warp < 2) {
      const int o = 32 * warp;
      float* W = Wt + 16 * warp * LDW;  // this warp's 16 x 16 part of the buffer
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        mma_f32x3(acc, As, LDF, o + 16, o, Tms, LDF, o, o + 8 * nt, lane);
        store_tile(W, LDW, 0, 8 * nt, acc, 1.f, lane);
      }
      __syncwarp();
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        mma_f32x3(acc, Tms, LDF, o + 16, o + 16, W, LDW, 0, 8 * nt, lane);
        store_tile(Tms, LDF, o + 16, o + 8 * nt, acc, -1.f, lane);
      }
    }
    __syncthreads();

    // ---- merge 32 -> 64: T[32.., 0..32] = -T[32..,32..] (A[32..,0..32] T[0..32,0..32]) ----
    {
      const int mt = warp >> 2, nt = warp & 3;
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int kk = 0; kk < 2; ++kk) mma_f32x3(acc, As, LDF, 32 + 16 * mt, 16 * kk, Tms, LDF, 16 * kk, 8 * nt, lane);
      store_tile(Wt, LDW, 16 * mt, 8 * nt, acc, 1.f, lane);
      __syncthreads();
      float acc2[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int kk = 0; kk < 2; ++kk)
        mma_f32x3(acc2, Tms, LDF, 32 + 16 * mt, 32 + 16 * kk, Wt, LDW, 16 * kk, 8 * nt, lane);
      store_tile(Tms, LDF, 32 + 16 * mt, 8 * nt, acc2, -1.f, lane);
    }
    __syncthreads();

    // ---- bf16 Tm: to shared (for PT) and to the workspace ---------------------
    __nv_bfloat16* wsT = ws + ((size_t)slot * Hv + h) * (2 * kWsTileElems);
    __nv_bfloat16* wsPT = wsT + kWsTileElems;
    for (int e = tid; e < kChunk * 8; e += kPrepThreads) {
      const int r = e >> 3, p = e & 7;
      const float* src = Tms + r * LDF + 8 * p;
      uint4 v;
      v.x = pack_bf16(src[0], src[1]);
      v.y = pack_bf16(src[2], src[3]);
      v.z = pack_bf16(src[4], src[5]);
      v.w = pack_bf16(src[6], src[7]);
      *reinterpret_cast<uint4*>(Tmb + r * LDB + 8 * p) = v;
      *reinterpret_cast<uint4*>(wsT + r * kChunk + 8 * p) = v;
    }
    __syncthreads();

    // ---- PT = P Tm (lower triangular); warp w: rows 16 (w/2).., column pairs ---
    {
      const int mi = warp >> 1, m = lane >> 3;
      float acc[4][4];
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        if (kk <= mi) {
          uint32_t a[4];
          ldsm_x4(a, Ps + (16 * mi + 8 * (m & 1) + (lane & 7)) * LDB + 16 * kk + 8 * (m >> 1));
#pragma unroll
          for (int pp = 0; pp < 2; ++pp) {
            const int p = 2 * (warp & 1) + pp;  // column pair: columns 16 p .. 16 p + 15
            if (p <= kk) {
              uint32_t bb[4];
              ldsm_x4_t(bb, Tmb + (16 * kk + 8 * (m & 1) + (lane & 7)) * LDB + 8 * (2 * p + (m >> 1)));
              mma_bf16(acc[2 * pp], a, bb[0], bb[1]);
              mma_bf16(acc[2 * pp + 1], a, bb[2], bb[3]);
            }
          }
        }
      }
      __syncthreads();  // every warp has read P before it is overwritten with PT
      const int r0 = 16 * mi + (lane >> 2);
#pragma unroll
      for (int pp = 0; pp < 2; ++pp) {
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int cc = 16 * (2 * (warp & 1) + pp) + 8 * hh + 2 * (lane & 3);
          *reinterpret_cast<uint32_t*>(Ps + r0 * LDB + cc) = pack_bf16(acc[2 * pp + hh][0], acc[2 * pp + hh][1]);
          *reinterpret_cast<uint32_t*>(Ps + (r0 + 8) * LDB + cc) =
              pack_bf16(acc[2 * pp + hh][2], acc[2 * pp + hh][3]);
        }
      }
    }
    __syncthreads();
    for (int e = tid; e < kChunk * 8; e += kPrepThreads) {
      const int r = e >> 3, p = e & 7;
      *reinterpret_cast<uint4*>(wsPT + r * kChunk + 8 * p) =
          *reinterpret_cast<const uint4*>(Ps + r * LDB + 8 * p);
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
  gdn_prep_kernel<DK><<<grid, kPrepThreads, L::bytes, st>>>(
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
