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
// once per key head (one tcgen05 product in TMEM).  The inverse is blocked: the
// four 16 x 16 diagonal blocks by forward substitution in fp32, then the
// 16 -> 32 -> 64 merges T21 = -T22 A21 T11 as tensor-core products whose fp32
// operands are split into bf16 hi + lo parts (hi*hi + hi*lo + lo*hi, ~2^-16
// relative).  Only non-positive exponents are ever taken (gamma_t - gamma_i,
// i <= t), so nothing overflows however strong the decay.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "gdn_tc.cuh"

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
  // [union: K,Q tiles (TMA, 128 B swizzle) | A,Tm fp32] [G fp32 x2] [P bf16] [Tm bf16] [merge buffer]
  // [inverse norms] [g, beta] [mbarriers]
  static constexpr int kKQBytes = 32768;
  static constexpr int kATBytes = 2 * kChunk * LDF * 4;
  static constexpr int kUnion = kKQBytes > kATBytes ? kKQBytes : kATBytes;
  static constexpr int offG = kUnion;
  static constexpr int offP = offG + 2 * kChunk * LDF * 4;
  static constexpr int offTb = offP + kChunk * LDB * 2;
  static constexpr int offW = offTb + kChunk * LDB * 2;
  static constexpr int offRN = offW + 32 * LDW * 4;  // inverse norms of k rows, then q rows
  static constexpr int offGB = offRN + 2 * kChunk * 4;   // [2 buffers][g 64 | beta 64] fp32
  static constexpr int offBar = offGB + 2 * 2 * kChunk * 4;
  static constexpr int bytes = offBar + 32 + 1024;  // 2 mbarriers + TMEM base; + slack for 1024-byte alignment
};

template <int DK>
__global__ void __launch_bounds__(kPrepThreads, 2)
gdn_prep_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_q,
                const float* __restrict__ g, const float* __restrict__ beta,
                const int32_t* __restrict__ cu, const int32_t* __restrict__ chunk_off,
                __nv_bfloat16* __restrict__ ws, float* __restrict__ ws_rn, int* __restrict__ err, int B,
                int T, int Hk, int Hv, int nc_dense, int norm_qk, int hk_base, int hk_count, int c_begin,
                int c_count, int n_items) {
  using L = PrepSmem<DK>;
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw_s = smem_u32(smem_raw);
  unsigned char* smem = smem_raw + (((raw_s + 1023u) & ~1023u) - raw_s);
  unsigned char* KQ = smem;                    // [2][128][128 B], swizzled
  float* As = reinterpret_cast<float*>(smem);  // aliases K/Q after the Grams
  float* Tms = As + kChunk * LDF;
  float* Gs = reinterpret_cast<float*>(smem + L::offG);  // [2][64][LDF]
  __nv_bfloat16* Ps = reinterpret_cast<__nv_bfloat16*>(smem + L::offP);
  __nv_bfloat16* Tmb = reinterpret_cast<__nv_bfloat16*>(smem + L::offTb);
  float* Wt = reinterpret_cast<float*>(smem + L::offW);  // [32][LDW]
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + L::offBar);  // [0] tiles loaded, [1] Grams done
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::offBar + 16);
  float* gbuf = reinterpret_cast<float*>(smem + L::offGB);
  float* rnk = reinterpret_cast<float*>(smem + L::offRN);  // 1/||k_t|| (1 without normalisation)
  float* rnq = rnk + kChunk;                                // 1/||q_t||

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int kKBlocks = DK > 64 ? 2 : 1;
  constexpr uint32_t kGramCols = 64;
  const int G = Hv / Hk;

  // Items are (chunk slot, key head) pairs: item = x * hk_count + (key head - hk_base).  Dense
  // batches: slot index x is chunk c_begin + x % c_count of sequence x / c_count (a window of
  // each sequence's chunks; the whole sequence when c_begin = 0, c_count = nc_dense).  Packed
  // batches: x is the slot, and slots past the last chunk are empty.
  struct Item {
    int slot, hk, b, c, n;
    long long t0;
  };
  auto locate = [&](int item, Item& it) -> bool {
    const int x = item / hk_count;
    it.hk = hk_base + (item - x * hk_count);
    if (cu == nullptr) {
      it.b = x / c_count;
      it.c = c_begin + (x - it.b * c_count);
      if (it.b >= B) return false;
      it.slot = it.b * nc_dense + it.c;
    } else {
      if (x >= chunk_off[B]) return false;
      int lo = 0, hi = B;  // largest b with chunk_off[b] <= x
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (chunk_off[mid] <= x) lo = mid; else hi = mid;
      }
      it.b = lo;
      it.c = x - chunk_off[lo];
      it.slot = x;
    }
    const SeqChunk sq = seq_bounds(cu, it.b, T);
    it.t0 = sq.bos + (long long)it.c * kChunk;
    it.n = min(kChunk, sq.len - it.c * kChunk);
    return true;
  };

  // g and beta of value head gi of an item into buffer `buf` (zeros past the chunk's
  // tokens), by warps 2 and 3, beside thread 0's copies
  auto load_gb = [&](const Item& it, int gi, int buf) {
    const int lt = tid - 64;
    if (lt >= 0 && lt < kChunk) {
      const bool ok = lt < it.n;
      const size_t off = ok ? (size_t)(it.t0 + lt) * Hv + it.hk * G + gi : 0;
      cp_async4(gbuf + buf * 2 * kChunk + lt, g + off, ok);
      cp_async4(gbuf + buf * 2 * kChunk + kChunk + lt, beta + off, ok);
    }
    cp_async_commit();
  };
  // An item's K and Q tiles by TMA (tokens past the end are zero), and the tiles of the
  // CTA's following item into L2 (thread 0)
  auto load_tiles = [&](int item, const Item& it) {
    tc::mbar_arrive_expect_tx(&bar[0], 2 * kKBlocks * 8192);
#pragma unroll
    for (int db = 0; db < kKBlocks; ++db) {
      tc::tma_load_3d(KQ + db * 16384, &tm_k, 64 * db, it.hk, (int)it.t0, &bar[0]);
      tc::tma_load_3d(KQ + db * 16384 + 8192, &tm_q, 64 * db, it.hk, (int)it.t0, &bar[0]);
    }
    Item nx;
    if (item + (int)gridDim.x < n_items && locate(item + (int)gridDim.x, nx)) {
#pragma unroll
      for (int db = 0; db < kKBlocks; ++db) {
        tc::tma_prefetch_l2_3d(&tm_k, 64 * db, nx.hk, (int)nx.t0);
        tc::tma_prefetch_l2_3d(&tm_q, 64 * db, nx.hk, (int)nx.t0);
      }
    }
  };

  // ---- once per CTA: barriers, TMEM for the Grams; the first item's loads beside them ---
  Item first;
  const bool first_ok = locate(blockIdx.x, first);
  if (tid == 0) {
    tc::prefetch_tensormap(&tm_k);
    tc::prefetch_tensormap(&tm_q);
    tc::mbar_init(&bar[0], 1);
    tc::mbar_init(&bar[1], 1);
    tc::fence_mbar_init();
    if (first_ok) load_tiles(blockIdx.x, first);
  }
  if (first_ok) load_gb(first, 0, 0);
  if (warp == 1) {
    tc::tmem_alloc(tmem_slot, kGramCols);
    tc::tmem_relinquish();
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = *tmem_slot;

  // Persistent CTAs (two per SM) walk the items with the grid's stride.  While one item is
  // worked on, the next one's key and query tiles are brought into L2, so its tile copy
  // does not wait for DRAM.
  uint32_t ph = 0;  // phase of bar[0] and bar[1]: each completes once per item worked on
  for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
    Item cur;
    if (!locate(item, cur)) continue;  // the same for every thread of the CTA
    const int slot = cur.slot, hk = cur.hk, n = cur.n;

    // the loads of this item (the first item's went out before the set-up barrier)
    if (item != (int)blockIdx.x) {
      load_gb(cur, 0, 0);
      if (tid == 0) load_tiles(item, cur);
    }
    if (!tc::mbar_wait(&bar[0], ph, 1u << 24)) atomicOr(err, 4);
    // rows t >= n belong to the next sequence (or are past the end): clear them
    if (n < kChunk) {
      for (int e = tid; e < kKBlocks * 2 * (kChunk - n) * 8; e += kPrepThreads) {
        const int piece = e & 7, rr = e >> 3;
        const int r = n + rr % (kChunk - n), which = (rr / (kChunk - n)) & 1, db = rr / (2 * (kChunk - n));
        *reinterpret_cast<uint4*>(KQ + db * 16384 + tc::sw128(64 * which + r, piece)) = make_uint4(0, 0, 0, 0);
      }
    }
    tc::fence_proxy_async();  // the cleared rows are read by the tensor core
    __syncthreads();

    // ---- Grams on the tensor core: D = [K; Q] K^T (M = 128, N = 64, K = dk) -------
    // Rows 0..63 of D are K K^T, rows 64..127 Q K^T; both operands are the K-major
    // swizzled tile as loaded (the B operand is its first 64 rows).
    if (tid == 0) {
      tc::fence_after();
      constexpr uint32_t kID = tc::idesc_bf16(128, 64, 0, 0);
      const uint32_t kq = smem_u32(KQ);
#pragma unroll
      for (int ks = 0; ks < DK / 16; ++ks) {
        const uint32_t off = (ks >> 2) * 16384 + (ks & 3) * 32;
        tc::mma_bf16(tmem, tc::sdesc(kq + off, 16, 1024, tc::kSw128), tc::sdesc(kq + off, 16, 1024, tc::kSw128), kID,
                     ks > 0);
      }
      tc::commit(&bar[1]);
    }
    // inverse norms of the k and q rows while the product runs
    if (tid < 2 * kChunk) {
      const float r = norm_qk ? tc::inv_norm(tc::row_sumsq_sw128<DK>(KQ, (tid & 63) + 64 * (tid >> 6))) : 1.f;
      rnk[tid] = r;  // tid 0..63: k rows, 64..127: q rows (rnq = rnk + 64)
      if (norm_qk) ws_rn[((size_t)slot * Hk + hk) * (2 * kChunk) + tid] = r;  // for the state carry
    }
    if (!tc::mbar_wait(&bar[1], ph, 1u << 24)) atomicOr(err, 4);
    tc::fence_after();
    // TMEM -> the fp32 Grams: warp w reads lanes 32 (w % 4) .. +31 (rows: 0..63 K, 64..127
    // Q) and columns 32 (w / 4) .. +31
    {
      const int q4 = warp & 3, hf = warp >> 2;
      float v[32];
      tc::tmem_ld32(tmem + ((uint32_t)(32 * q4) << 16) + 32 * hf, v);
      float* dst = Gs + (q4 >> 1) * kChunk * LDF + (32 * (q4 & 1) + lane) * LDF + 32 * hf;
#pragma unroll
      for (int p = 0; p < 8; ++p)
        *reinterpret_cast<float4*>(dst + 4 * p) = make_float4(v[4 * p], v[4 * p + 1], v[4 * p + 2], v[4 * p + 3]);
    }
    tc::fence_before();
    __syncthreads();  // Grams and norms visible; the tiles are dead from here on (A and Tm overwrite them)


    for (int gi = 0; gi < G; ++gi) {
      const int h = hk * G + gi;
      // this head's g / beta arrived by cp.async; start fetching the next head's
      cp_async_wait<0>();
      __syncthreads();
      if (gi + 1 < G) load_gb(cur, gi + 1, (gi + 1) & 1);
      // ---- gamma = inclusive cumsum of g in the chunk, in log2 units -------------------
      // Every warp scans the 64 values in registers (lane l holds tokens l and l + 32), so
      // no warp waits for another; the A/P build below takes its entries by shuffle.
      const float* gb = gbuf + (gi & 1) * 2 * kChunk;  // [g 64 | beta 64]
      float gl0 = gb[lane], gl1 = gb[lane + 32];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float u0 = __shfl_up_sync(0xffffffffu, gl0, o);
        const float u1 = __shfl_up_sync(0xffffffffu, gl1, o);
        if (lane >= o) { gl0 += u0; gl1 += u1; }
      }
      gl1 += __shfl_sync(0xffffffffu, gl0, 31);
      gl0 *= 1.4426950408889634f;  // log2(e)
      gl1 *= 1.4426950408889634f;

      // ---- A (fp32) and P (bf16), 8 columns at a time, lower triangle only ----------
      // Gamma[t][i] = 2^(gamma2_t - gamma2_i) with gamma2 = gamma log2(e): the exponent
      // is never positive for i <= t.  A thread keeps one 8-column block (the CTA size is
      // a multiple of 8), so its gamma and 1/||k|| columns are loaded once.
      static_assert(kPrepThreads == 256, "two (row, column block) items per thread, rows tid / 8 and + 32");
      const int c8 = (tid & 7) * 8;
      float gcol[8], rcol[8];
      {
#pragma unroll
        for (int u = 0; u < 8; ++u) {  // gamma of columns c8 .. c8 + 7 (tokens < 32 in gl0, the rest in gl1)
          const float lo = __shfl_sync(0xffffffffu, gl0, (c8 + u) & 31);
          const float hi = __shfl_sync(0xffffffffu, gl1, (c8 + u) & 31);
          gcol[u] = c8 < 32 ? lo : hi;
        }
        const float4 r0 = *reinterpret_cast<const float4*>(rnk + c8), r1 = *reinterpret_cast<const float4*>(rnk + c8 + 4);
        rcol[0] = r0.x; rcol[1] = r0.y; rcol[2] = r0.z; rcol[3] = r0.w;
        rcol[4] = r1.x; rcol[5] = r1.y; rcol[6] = r1.z; rcol[7] = r1.w;
      }
      // gamma of this thread's two rows, tid / 8 and tid / 8 + 32 (lane (tid / 8) % 32 of this warp)
      const float grow0 = __shfl_sync(0xffffffffu, gl0, (tid >> 3) & 31);
      const float grow1 = __shfl_sync(0xffffffffu, gl1, (tid >> 3) & 31);
      for (int e = tid; e < kChunk * 8; e += kPrepThreads) {
        const int t = e >> 3;
        float av[8], pv[8];
        if (c8 <= t) {
          const float gt = t < 32 ? grow0 : grow1, bt = gb[kChunk + t] * rnk[t], qt = rnq[t];
          const float4 k0 = *reinterpret_cast<const float4*>(Gs + t * LDF + c8);
          const float4 k1 = *reinterpret_cast<const float4*>(Gs + t * LDF + c8 + 4);
          const float4 q0 = *reinterpret_cast<const float4*>(Gs + kChunk * LDF + t * LDF + c8);
          const float4 q1 = *reinterpret_cast<const float4*>(Gs + kChunk * LDF + t * LDF + c8 + 4);
          const float gk[8] = {k0.x, k0.y, k0.z, k0.w, k1.x, k1.y, k1.z, k1.w};
          const float gq[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const int i = c8 + u;
            const float dcy = i <= t ? exp2f(gt - gcol[u]) * rcol[u] : 0.f;
            pv[u] = qt * dcy * gq[u];
            av[u] = i < t ? bt * dcy * gk[u] : 0.f;
          }
        } else {
#pragma unroll
          for (int u = 0; u < 8; ++u) av[u] = pv[u] = 0.f;
        }
        *reinterpret_cast<float4*>(As + t * LDF + c8) = make_float4(av[0], av[1], av[2], av[3]);
        *reinterpret_cast<float4*>(As + t * LDF + c8 + 4) = make_float4(av[4], av[5], av[6], av[7]);
        *reinterpret_cast<uint4*>(Ps + t * LDB + c8) =
            make_uint4(pack_bf16(pv[0], pv[1]), pack_bf16(pv[2], pv[3]), pack_bf16(pv[4], pv[5]),
                       pack_bf16(pv[6], pv[7]));
      }
      if (gi == 0) {  // the blocks of Tm above the diagonal stay zero for every value head
        for (int e = tid; e < kChunk * 16; e += kPrepThreads) {
          const int t = e >> 4, c4 = (e & 15) * 4;
          if ((c4 >> 4) > (t >> 4)) *reinterpret_cast<float4*>(Tms + t * LDF + c4) = make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
      __syncthreads();

      // ---- Tm: the four 16 x 16 diagonal blocks by forward substitution --------
      // Column j of a block: x_j = 1, then for i = j, j+1, ...: x_{i+1} = -acc_{i+1}
      // after every later acc_t has absorbed A[t][i] x_i (right-looking order, so
      // the dependent chain is one FMA per row).
      if (tid < 64) {
        const int blk = tid >> 4, j = tid & 15;
        const float* Ab = As + 16 * blk * LDF + 16 * blk;
        float x[16], accv[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) { x[i] = (i == j) ? 1.f : 0.f; accv[i] = 0.f; }
#pragma unroll
        for (int i = 0; i < 15; ++i) {
          if (i > j) x[i] = -accv[i];
#pragma unroll
          for (int t = i + 1; t < 16; ++t) accv[t] = fmaf(Ab[t * LDF + i], x[i], accv[t]);
        }
        if (15 > j) x[15] = -accv[15];
        float* Tb = Tms + 16 * blk * LDF + 16 * blk;
#pragma unroll
        for (int t = 0; t < 16; ++t) Tb[t * LDF + j] = x[t];
      }
      __syncthreads();

      // ---- merge 16 -> 32: T[o+16.., o..] = -T22 (A21 T11), o = 0 and 32 -------
      // Warp w < 4 forms the 8-column tile nt = w % 2 of block o = 32 (w / 2): its column
      // tile of W = A21 T11 is all that its tile of T21 = -T22 W needs.
      if (warp < 4) {
        const int o = 32 * (warp >> 1), nt = warp & 1;
        float* W = Wt + 16 * (warp >> 1) * LDW;  // this block's 16 x 16 part of the buffer
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        mma_f32x3(acc, As, LDF, o + 16, o, Tms, LDF, o, o + 8 * nt, lane);
        store_tile(W, LDW, 0, 8 * nt, acc, 1.f, lane);
        __syncwarp();
        float acc2[4] = {0.f, 0.f, 0.f, 0.f};
        mma_f32x3(acc2, Tms, LDF, o + 16, o + 16, W, LDW, 0, 8 * nt, lane);
        store_tile(Tms, LDF, o + 16, o + 8 * nt, acc2, -1.f, lane);
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
    ph ^= 1;
    tc::fence_proxy_async();  // the next item's tile copy overwrites what this one left in shared memory
    __syncthreads();
  }
  if (warp == 1) tc::tmem_dealloc(tmem, kGramCols);
}

// Prefix sums of chunk counts for packed sequences: chunk_off[b] = sum over
// b' < b of ceil(len_b' / 64), chunk_off[B] = total.  One CTA of 1024 threads.  It also
// checks cu_seqlens (0 = cu[0] <= cu[1] <= ... <= cu[B] = T) and records status bit 8 when
// the array is malformed; every kernel clamps the entries to [0, T] all the same.
__global__ void __launch_bounds__(1024)
gdn_chunk_table_kernel(const int32_t* __restrict__ cu, int B, int T, int32_t* __restrict__ chunk_off,
                       int* __restrict__ err) {
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
      const int lo = cu[b], hi = cu[b + 1];
      if (lo < 0 || hi < lo || hi > T || (b == 0 && lo != 0) || (b == B - 1 && hi != T)) atomicOr(err, 8);
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
namespace {
PFN_cuTensorMapEncodeTiled_v12000 prep_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (fn == nullptr) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult qr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &qr) ==
            cudaSuccess &&
        qr == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}
}  // namespace

template <int DK>
cudaError_t launch_prep(const void* q, const void* k, const float* g, const float* beta,
                        const int32_t* cu, const int32_t* chunk_off, void* ws, float* ws_rn, int* err, int B, int T,
                        int Hk, int Hv, int nslots, int nc_dense, int norm_qk, int hk_base, int hk_count,
                        int c_begin, int c_count, int persistent, cudaStream_t st) {
  using L = PrepSmem<DK>;
  PFN_cuTensorMapEncodeTiled_v12000 enc = prep_map_encoder();
  if (enc == nullptr) return cudaErrorNotSupported;
  const long long ttot = cu != nullptr ? (long long)T : (long long)B * T;
  const cuuint64_t dims[3] = {(cuuint64_t)DK, (cuuint64_t)Hk, (cuuint64_t)(ttot > 0 ? ttot : 1)};
  const cuuint64_t strides[2] = {(cuuint64_t)DK * 2, (cuuint64_t)Hk * DK * 2};
  const cuuint32_t box[3] = {64, 1, 64}, es[3] = {1, 1, 1};
  CUtensorMap mk, mq;
  if (enc(&mk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(k), dims, strides, box, es,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS ||
      enc(&mq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(q), dims, strides, box, es,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  cudaError_t e = set_smem_limit_once<gdn_prep_kernel<DK>>(L::bytes);
  if (e != cudaSuccess) return e;
  if (cu == nullptr && (c_begin < 0 || c_count <= 0 || c_begin + c_count > nc_dense)) return cudaErrorInvalidValue;
  // items: key heads hk_base .. hk_base + hk_count - 1 of B sequences x c_count chunks (dense)
  // or of every slot (packed).  With the device to itself: persistent CTAs, two per SM.  Beside
  // other kernels (the host entry's pipelines) a CTA per item, so that the hardware spreads the
  // items over whatever SMs come free.
  const long long n_items = (cu == nullptr ? (long long)B * c_count : (long long)nslots) * hk_count;
  if (n_items <= 0) return cudaSuccess;
  if (n_items > 0x7fffffffLL) return cudaErrorInvalidValue;
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess ||
      (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
    return e;
  const long long grid = persistent && n_items > 2LL * sms ? 2LL * sms : n_items;
  gdn_prep_kernel<DK><<<(unsigned)grid, kPrepThreads, L::bytes, st>>>(mk, mq, g, beta, cu, chunk_off,
                                                           static_cast<__nv_bfloat16*>(ws), ws_rn, err, B, T, Hk, Hv,
                                                           nc_dense, norm_qk, hk_base, hk_count, c_begin,
                                                           c_count, (int)n_items);
  return cudaGetLastError();
}

cudaError_t launch_chunk_table(const int32_t* cu, int B, int T, int32_t* chunk_off, int* err, cudaStream_t st) {
  gdn_chunk_table_kernel<<<1, 1024, 0, st>>>(cu, B, T, chunk_off, err);
  return cudaGetLastError();
}

#define GDN_INST_PREP(DK)                                                                                  \
  template cudaError_t launch_prep<DK>(const void*, const void*, const float*, const float*, const int32_t*, \
                                       const int32_t*, void*, float*, int*, int, int, int, int, int, int, int,  \
                                       int, int, int, int, int, cudaStream_t);
GDN_INST_PREP(32)
GDN_INST_PREP(64)
GDN_INST_PREP(128)

}  // namespace gdn
