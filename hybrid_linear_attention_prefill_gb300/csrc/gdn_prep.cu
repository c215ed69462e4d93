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
// Tm and PT are stored as 64 x 64 tiles in the workspace -- bf16 for the wide-range
// state carry; for the default one fp16, with Tm's rows scaled by d_t = exp(gamma_last -
// gamma_t), the diag(d) Tm of its W = K^T diag(d) Tm -- and the state-carry kernel
// combines them with the state.  For the fp16 state carry the kernel also writes the chunk's
// k and q rows as fp16 (normalised when asked to), since a tensor-core product takes
// both operands in one format.  The pages only name the operation (the
// "chunked Gated DeltaNet prefill" of the "Open-Jev-27B-v1.1 native text
// worker" page, "Validation and optimization scope"); the WY form is the
// standard chunked rewriting of S_t = a_t S_{t-1}(I - b_t k_t k_t^T) + b_t v_t k_t^T.
//
// One CTA (8 warps) handles one chunk slot and one key head, and loops over the
// value heads that share the key head, so the Grams K K^T and Q K^T are computed
// once per key head (one tcgen05 product in TMEM).  The inverse is blocked: the
// four 16 x 16 diagonal blocks by forward substitution in fp32, then the
// 16 -> 32 -> 64 merges T21 = -T22 A21 T11 as tensor-core products of fp16 blocks
// (each rounded once, when it is formed; fp32 accumulate).  Only non-positive exponents
// are ever taken (gamma_t - gamma_i, i <= t), so nothing overflows however strong the decay.
#include <atomic>
#include <cuda_fp16.h>
#include "gdn_tc.cuh"
#include "gdn_tmap.cuh"

namespace gdn {

namespace {

constexpr int kPrepThreads = 256;
constexpr int kPrepCtasPerSm = 4;  // resident CTAs per SM: registers by the launch bounds, shared memory below
constexpr int LDB = 72;   // 16-bit row stride of 64-wide matrices (144 B: ldmatrix rows on distinct banks)
constexpr int LDWH = 40;  // 16-bit row stride of the 32-wide merge buffer (80 B, likewise)
constexpr int LDD = 20;   // fp32 row stride of A's 16 x 16 diagonal blocks
// ... and the stride between those blocks: 16 banks apart, so the substitution's two blocks per
// warp (one per half-warp, every lane of a half reading the same entry) take one wavefront
constexpr int kDiagStride = 16 * LDD + 16;
constexpr int LDE = 20;   // fp32 row stride of the 16-wide decay tables

__device__ __forceinline__ uint32_t pack_f16(float a, float b) {
  __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

// Two values as the 16-bit format of the stored tiles: fp16 or bf16.
template <bool F16>
__device__ __forceinline__ uint32_t pack16(float a, float b) {
  if constexpr (F16) return pack_f16(a, b);
  else return pack_bf16(a, b);
}

// d += a b for one m16n8k16 fragment triple (ldmatrix layouts) of fp16 or bf16 values.
template <bool F16>
__device__ __forceinline__ void mma16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  if constexpr (F16) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  } else {
    mma_bf16(d, a, b0, b1);
  }
}

// ldmatrix for the merges' fp16 operands (the memory clobber keeps them after the stores they read)
__device__ __forceinline__ void ldsm_a(uint32_t (&r)[4], const uint16_t* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(p))
               : "memory");
}
__device__ __forceinline__ void ldsm_b_t(uint32_t (&r)[4], const uint16_t* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(p))
               : "memory");
}
__device__ __forceinline__ void ldsm_b8_t(uint32_t (&r)[2], const uint16_t* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0,%1}, [%2];\n"
               : "=r"(r[0]), "=r"(r[1])
               : "r"(smem_u32(p))
               : "memory");
}

// The m16n8k16 A fragment of the 16 x 16 fp16 block at X[r0.., k0..] (row stride ld), and the
// B fragment of the 16 x 8 block at Y[k0.., n0..] (row-major, k rows).
__device__ __forceinline__ void frag_a(uint32_t (&a)[4], const uint16_t* X, int ld, int r0, int k0, int lane) {
  const int m = lane >> 3;
  ldsm_a(a, X + (r0 + 8 * (m & 1) + (lane & 7)) * ld + k0 + 8 * (m >> 1));
}
__device__ __forceinline__ void frag_b8(uint32_t (&b)[2], const uint16_t* Y, int ld, int k0, int n0, int lane) {
  ldsm_b8_t(b, Y + (k0 + (lane & 15)) * ld + n0);
}

// Store a 16 x 8 accumulator tile (times `sgn`), rounded to fp16, at D[r0.., n0..].
__device__ __forceinline__ void store_tile_h(uint16_t* D, int ldd, int r0, int n0, const float (&acc)[4], float sgn,
                                             int lane) {
  const int g8 = lane >> 2, tg = lane & 3;
  *reinterpret_cast<uint32_t*>(D + (r0 + g8) * ldd + n0 + 2 * tg) = pack_f16(sgn * acc[0], sgn * acc[1]);
  *reinterpret_cast<uint32_t*>(D + (r0 + g8 + 8) * ldd + n0 + 2 * tg) = pack_f16(sgn * acc[2], sgn * acc[3]);
}

}  // namespace

template <int DK>
struct PrepSmem {
  // [union: K,Q tiles (TMA, 128 B swizzle) | the inverse's working set] [P 16-bit]
  // [Tm 16-bit | decay tables] [inverse norms] [column factors] [g, beta] [mbarriers]
  // (the Grams stay in TMEM; the CTA fits four times on an SM).  The working set of the inverse
  // -- A's blocks below the diagonal and Tm in fp16 (the merges' operands, each rounded once),
  // A's diagonal blocks in fp32 (the forward substitution), the fp16 merge buffer -- lives over
  // the key and query tiles, which are dead once the Grams and the image are done.  Within a
  // value head the decay tables live until A and P are built and the 16-bit Tm from then on, so
  // the two share one region.
  static constexpr int kKQBytes = 32768;
  static constexpr int offAh = 0;                          // [64][LDB] fp16
  static constexpr int offTh = offAh + kChunk * LDB * 2;   // [64][LDB] fp16
  static constexpr int offAd = offTh + kChunk * LDB * 2;   // [4][16][LDD] fp32, blocks kDiagStride apart
  static constexpr int offWh = offAd + 4 * kDiagStride * 4;  // [32][LDWH] fp16
  static constexpr int kMergeBytes = offWh + 32 * LDWH * 2;
  static constexpr int kUnion = kKQBytes > kMergeBytes ? kKQBytes : kMergeBytes;
  static constexpr int offP = kUnion;
  static constexpr int offTb = offP + kChunk * LDB * 2;
  static constexpr int offRN = offTb + kChunk * LDB * 2;  // inverse norms of k rows, then q rows
  static_assert(4 * 16 * LDE * 4 + kChunk * 4 * 4 <= kChunk * LDB * 2, "the decay tables fit over the 16-bit Tm");
  static constexpr int offCF = offRN + 2 * kChunk * 4;  // column factors [64]
  static constexpr int offGB = offCF + kChunk * 4;       // [2 buffers][g 64 | beta 64] fp32
  static constexpr int offBar = offGB + 2 * 2 * kChunk * 4;
  static constexpr int bytes = offBar + 32 + 1024;  // 2 mbarriers + TMEM base; + slack for 1024-byte alignment
};

// F16: Tm, P and PT in fp16, and the fp16 [K; Q] image for the state carry (ws_kq); else bf16.
template <int DK, bool F16>
__global__ void __launch_bounds__(kPrepThreads, kPrepCtasPerSm)
gdn_prep_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_q,
                const float* __restrict__ g, const float* __restrict__ beta,
                const int32_t* __restrict__ cu, const int32_t* __restrict__ chunk_off,
                uint16_t* __restrict__ ws, float* __restrict__ ws_rn, unsigned char* __restrict__ ws_kq,
                int* __restrict__ err, int B,
                int T, int Hk, int Hv, int nc_dense, int norm_qk, int hk_base, int hk_count, int c_begin,
                int c_count, int n_items) {
  using L = PrepSmem<DK>;
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw_s = smem_u32(smem_raw);
  unsigned char* smem = smem_raw + (((raw_s + 1023u) & ~1023u) - raw_s);
  unsigned char* KQ = smem;                    // [2][128][128 B], swizzled
  // the inverse's working set, over K / Q after the Grams
  uint16_t* Ah = reinterpret_cast<uint16_t*>(smem + L::offAh);  // A below its diagonal blocks, fp16
  uint16_t* Th = reinterpret_cast<uint16_t*>(smem + L::offTh);  // Tm, fp16
  float* Ad = reinterpret_cast<float*>(smem + L::offAd);         // A's diagonal blocks, fp32
  uint16_t* Wh = reinterpret_cast<uint16_t*>(smem + L::offWh);  // merge buffer, fp16
  uint16_t* Ps = reinterpret_cast<uint16_t*>(smem + L::offP);
  uint16_t* Tmb = reinterpret_cast<uint16_t*>(smem + L::offTb);
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + L::offBar);  // [0] tiles loaded, [1] Grams done
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::offBar + 16);
  float* gbuf = reinterpret_cast<float*>(smem + L::offGB);
  float* rnk = reinterpret_cast<float*>(smem + L::offRN);  // 1/||k_t|| (1 without normalisation)
  float* rnq = rnk + kChunk;                                // 1/||q_t||
  float* cfs = reinterpret_cast<float*>(smem + L::offCF);  // 1/||k_i|| 2^(gamma2_{i | 15} - gamma2_i)
  // Decay tables of a value head, over the 16-bit Tm (not in use while A and P are built):
  // Es[b][r][c] = 2^(gamma2_{16b+r} - gamma2_{16b+c}) / ||k_{16b+c}|| for c <= r (else 0), and
  // rfs[b][t] = 2^(gamma2_t - gamma2_{16b+15}) for the blocks b below t's own
  float* Es = reinterpret_cast<float*>(smem + L::offTb);  // [4][16][LDE]
  float* rfs = Es + 4 * 16 * LDE;                          // [4][64]

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

  // Persistent CTAs (as many per SM as fit) walk the items with the grid's stride.  While one item is
  // worked on, the next one's key and query tiles are brought into L2, so its tile copy
  // does not wait for DRAM.
  int cur_slot = 0, cur_hk = 0;  // the item write_kq_image writes
  // ---- fp16 [K; Q] for the state carry: the tile's image, row by row scaled by its inverse
  // norm when q and k are normalised in-kernel.  bf16 values of magnitude 2^-17 .. 65504 are
  // exact in fp16.  Byte 16 e of the image lies in tile row (e / 8) % 128 wherever the swizzle
  // puts it in the row, so the image is copied in order.
  auto write_kq_image = [&](bool scaled) {
    if constexpr (F16) {
      unsigned char* dst = ws_kq + ((size_t)cur_slot * Hk + cur_hk) * kws_kq_bytes(DK);
      for (int e = tid; e < kKBlocks * 1024; e += kPrepThreads) {
        const float sc = scaled ? rnk[(e >> 3) & 127] : 1.f;  // k rows 0..63, then q rows (rnq = rnk + 64)
        const uint4 raw = *reinterpret_cast<const uint4*>(KQ + 16 * e);
        const uint32_t w4[4] = {raw.x, raw.y, raw.z, raw.w};
        uint32_t o4[4];
#pragma unroll
        for (int p = 0; p < 4; ++p)
          o4[p] = pack_f16(sc * __uint_as_float(w4[p] << 16), sc * __uint_as_float(w4[p] & 0xffff0000u));
        *reinterpret_cast<uint4*>(dst + 16 * e) = make_uint4(o4[0], o4[1], o4[2], o4[3]);
      }
    }
  };
  uint32_t ph = 0;  // phase of bar[0] and bar[1]: each completes once per item worked on
  int ahead = -1;   // (thread 0) the item whose tiles went out while the one before it was worked on
  for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
    Item cur;
    if (!locate(item, cur)) continue;  // the same for every thread of the CTA
    const int slot = cur.slot, hk = cur.hk, n = cur.n;
    cur_slot = slot;
    cur_hk = hk;

    // the loads of this item (the first item's went out before the set-up barrier)
    if (item != (int)blockIdx.x) {
      load_gb(cur, 0, 0);
      if (tid == 0 && item != ahead) load_tiles(item, cur);
    }
    // Thread 0 issued the tile copies and waits for them; the barriers below publish the tiles
    // to the other threads (a barrier makes the accesses a thread requested and saw complete
    // visible to all), so 255 more waits on the same phase are not needed.
    if (tid == 0 && !tc::mbar_wait(&bar[0], ph, 1u << 24)) atomicOr(err, 4);
    // rows t >= n belong to the next sequence (or are past the end): clear them once the copy is in
    if (n < kChunk) {
      __syncthreads();
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
      if (norm_qk && !F16) ws_rn[((size_t)slot * Hk + hk) * (2 * kChunk) + tid] = r;  // for the state carry
    }
    // without normalisation the image needs no norms: written while the product runs (the
    // tensor core only reads the tile)
    if (F16 && !norm_qk) write_kq_image(false);
    if (tid == 0 && !tc::mbar_wait(&bar[1], ph, 1u << 24)) atomicOr(err, 4);  // its own MMAs' commit
    tc::fence_before();
    __syncthreads();  // Grams done (they stay in TMEM) and norms visible; the tiles are dead after the image
    tc::fence_after();

    if (F16 && norm_qk) write_kq_image(true);  // scaled by the norms just summed

    for (int gi = 0; gi < G; ++gi) {
      const int h = hk * G + gi;
      // this head's g / beta arrived by cp.async; start fetching the next head's
      cp_async_wait<0>();
      __syncthreads();
      if (gi + 1 < G) load_gb(cur, gi + 1, (gi + 1) & 1);
      // ---- gamma = inclusive cumsum of g in the chunk, in log2 units -------------------
      // Warp 0 scans the 64 values once (lane l: tokens 2l and 2l + 1, then a five-step warp
      // scan of the pair sums) and writes gamma2 over this head's g, which nothing reads
      // afterwards; every thread then takes the entries it needs from shared memory.
      float* gb = gbuf + (gi & 1) * 2 * kChunk;  // [g 64 | beta 64]; g becomes gamma2
      if (warp == 0) {
        const float2 gg = *reinterpret_cast<const float2*>(gb + 2 * lane);
        const float pair = gg.x + gg.y;
        float incl = pair;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const float u = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += u;
        }
        const float excl = incl - pair;
        *reinterpret_cast<float2*>(gb + 2 * lane) =
            make_float2((excl + gg.x) * 1.4426950408889634f, incl * 1.4426950408889634f);  // log2(e)
      }
      __syncthreads();
      const float* g2 = gb;  // gamma2 of the chunk's tokens

      // ---- the decay tables of this value head (every thread) ----------------------------
      // Gamma[t][i] = 2^(gamma2_t - gamma2_i), i <= t, with every exponent <= 0: inside a
      // 16 x 16 diagonal block from the table Es, below it as the product of a row factor
      // (to the block's last column j0) and a column factor (from j0), both <= 1.
      {
        static_assert(kPrepThreads == 256, "one table row block per 256 entries");
        const int r = (tid >> 4) & 15, c = tid & 15;
#pragma unroll
        for (int bl = 0; bl < 4; ++bl)  // Es[bl][r][c]
          Es[(16 * bl + r) * LDE + c] = c <= r ? exp2f(g2[16 * bl + r] - g2[16 * bl + c]) * rnk[16 * bl + c] : 0.f;
        {
          const int t = tid & 63, bl = tid >> 6;  // rfs[bl][t] = rfs[tid]
          rfs[tid] = bl < (t >> 4) ? exp2f(g2[t] - g2[16 * bl + 15]) : 0.f;
        }
        if (tid < kChunk) cfs[tid] = rnk[tid] * exp2f(g2[tid | 15] - g2[tid]);  // warps 0 and 1: tokens tid
      }
      __syncthreads();

      // ---- A and P (16-bit) straight from the Grams in TMEM ------------------------------
      // Warp w reads TMEM lanes 32 (w % 4) .. + 31 -- rows 0..63 of the Gram are K K^T (A),
      // rows 64..127 Q K^T (P) -- and columns 32 (w / 4) .. + 31, 16 at a time.  A row's
      // entries in a 16-column block are the Gram's times one factor per row and one per
      // column: from Es in the row's own block (one row of it per lane), from the row and
      // column factors below it.
      {
        const int q4 = warp & 3, hf = warp >> 2;
        const bool isA = q4 < 2;
        const int t = 32 * (q4 & 1) + lane;  // token of this row
        const float sc = isA ? gb[kChunk + t] * rnk[t] : rnq[t];  // beta_t / ||k_t|| or 1 / ||q_t||
#pragma unroll
        for (int sb = 0; sb < 2; ++sb) {
          const int cb = 32 * hf + 16 * sb;
          float o[16];
          const bool own = t >= cb && t < cb + 16, below = t >= cb + 16;
          if (cb <= 32 * (q4 & 1) + 31) {  // warp-uniform: some row of the warp reaches column cb
            float v[16];
            tc::tmem_ld16(tmem + ((uint32_t)(32 * q4) << 16) + cb, v);
            const float* fp = own ? Es + t * LDE : cfs + cb;  // column factors of this row
            const float s = own ? sc : below ? sc * rfs[(cb >> 4) * kChunk + t] : 0.f;
#pragma unroll
            for (int u = 0; u < 16; u += 4) {
              const float4 f = *reinterpret_cast<const float4*>(fp + u);
              o[u] = s * f.x * v[u];
              o[u + 1] = s * f.y * v[u + 1];
              o[u + 2] = s * f.z * v[u + 2];
              o[u + 3] = s * f.w * v[u + 3];
            }
            if (isA && own) {  // A is strictly lower triangular
#pragma unroll
              for (int u = 0; u < 16; ++u)
                if (cb + u == t) o[u] = 0.f;
            }
          } else {
#pragma unroll
            for (int u = 0; u < 16; ++u) o[u] = 0.f;
          }
          if (isA) {
            if (own) {  // the diagonal block in fp32, for the forward substitution
              float* arow = Ad + (cb >> 4) * kDiagStride + (t - cb) * LDD;
#pragma unroll
              for (int p = 0; p < 4; ++p)
                *reinterpret_cast<float4*>(arow + 4 * p) = make_float4(o[4 * p], o[4 * p + 1], o[4 * p + 2], o[4 * p + 3]);
            } else if (below) {  // fp16, the merges' operands (the blocks above are never read)
              uint16_t* arow = Ah + t * LDB + cb;
#pragma unroll
              for (int p = 0; p < 2; ++p)
                *reinterpret_cast<uint4*>(arow + 8 * p) =
                    make_uint4(pack_f16(o[8 * p], o[8 * p + 1]), pack_f16(o[8 * p + 2], o[8 * p + 3]),
                               pack_f16(o[8 * p + 4], o[8 * p + 5]), pack_f16(o[8 * p + 6], o[8 * p + 7]));
            }
          } else {
            uint16_t* prow = Ps + t * LDB + cb;
#pragma unroll
            for (int p = 0; p < 2; ++p)
              *reinterpret_cast<uint4*>(prow + 8 * p) =
                  make_uint4(pack16<F16>(o[8 * p], o[8 * p + 1]), pack16<F16>(o[8 * p + 2], o[8 * p + 3]),
                             pack16<F16>(o[8 * p + 4], o[8 * p + 5]), pack16<F16>(o[8 * p + 6], o[8 * p + 7]));
          }
        }
      }
      tc::fence_before();  // the TMEM reads are ordered before the next item's Gram product
      if (gi == 0) {  // the blocks of Tm above the diagonal stay zero for every value head
        for (int e = tid; e < kChunk * 8; e += kPrepThreads) {
          const int t = e >> 3, c8 = (e & 7) * 8;
          if ((c8 >> 4) > (t >> 4)) *reinterpret_cast<uint4*>(Th + t * LDB + c8) = make_uint4(0, 0, 0, 0);
        }
      }
      __syncthreads();

      // ---- Tm: the four 16 x 16 diagonal blocks by forward substitution --------
      // Column j of a block: x_j = 1, then for i = j, j+1, ...: x_{i+1} = -acc_{i+1}
      // after every later acc_t has absorbed A[t][i] x_i (right-looking order, so
      // the dependent chain is one FMA per row).
      if (tid < 64) {
        const int blk = tid >> 4, j = tid & 15;
        const float* Ab = Ad + blk * kDiagStride;
        float x[16], accv[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) { x[i] = (i == j) ? 1.f : 0.f; accv[i] = 0.f; }
#pragma unroll
        for (int i = 0; i < 15; ++i) {
          if (i > j) x[i] = -accv[i];
#pragma unroll
          for (int t = i + 1; t < 16; ++t) accv[t] = fmaf(Ab[t * LDD + i], x[i], accv[t]);
        }
        if (15 > j) x[15] = -accv[15];
        uint16_t* Tb = Th + 16 * blk * LDB + 16 * blk;  // fp16: the merges' operand and the 16-bit Tm
#pragma unroll
        for (int t = 0; t < 16; ++t) Tb[t * LDB + j] = __half_as_ushort(__float2half_rn(x[t]));
      }
      __syncthreads();

      // ---- merge 16 -> 32: T[o+16.., o..] = -T22 (A21 T11), o = 0 and 32 -------
      // Warp w < 4 forms the 8-column tile nt = w % 2 of block o = 32 (w / 2): its column
      // tile of W = A21 T11 is all that its tile of T21 = -T22 W needs.  Operands by ldmatrix
      // from the fp16 blocks; the products accumulate in fp32 and are rounded to fp16 once.
      if (warp < 4) {
        const int o = 32 * (warp >> 1), nt = warp & 1;
        uint16_t* W = Wh + 16 * (warp >> 1) * LDWH;  // this block's 16 x 16 part of the buffer
        uint32_t a[4], b[2];
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        frag_a(a, Ah, LDB, o + 16, o, lane);
        frag_b8(b, Th, LDB, o, o + 8 * nt, lane);
        mma16<true>(acc, a, b[0], b[1]);
        store_tile_h(W, LDWH, 0, 8 * nt, acc, 1.f, lane);
        __syncwarp();
        float acc2[4] = {0.f, 0.f, 0.f, 0.f};
        frag_a(a, Th, LDB, o + 16, o + 16, lane);
        frag_b8(b, W, LDWH, 0, 8 * nt, lane);
        mma16<true>(acc2, a, b[0], b[1]);
        store_tile_h(Th, LDB, o + 16, o + 8 * nt, acc2, -1.f, lane);
      }
      __syncthreads();

      // ---- merge 32 -> 64: T[32.., 0..32] = -T[32..,32..] (A[32..,0..32] T[0..32,0..32]) ----
      {
        const int mt = warp >> 2, nt = warp & 3;
        uint32_t a[4], b[2];
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {
          frag_a(a, Ah, LDB, 32 + 16 * mt, 16 * kk, lane);
          frag_b8(b, Th, LDB, 16 * kk, 8 * nt, lane);
          mma16<true>(acc, a, b[0], b[1]);
        }
        store_tile_h(Wh, LDWH, 16 * mt, 8 * nt, acc, 1.f, lane);
        __syncthreads();
        float acc2[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {
          frag_a(a, Th, LDB, 32 + 16 * mt, 32 + 16 * kk, lane);
          frag_b8(b, Wh, LDWH, 16 * kk, 8 * nt, lane);
          mma16<true>(acc2, a, b[0], b[1]);
        }
        store_tile_h(Th, LDB, 32 + 16 * mt, 8 * nt, acc2, -1.f, lane);
      }
      __syncthreads();

      // ---- 16-bit Tm: to shared (for PT) and to the workspace ------------------
      // fp16 as it stands for PT; the workspace tile of the fp16 state carry holds diag(d) Tm,
      // d_t = exp(gamma_last - gamma_t) (its W = K^T diag(d) Tm), each row rounded once more.
      // The wide-range path's bf16 Tm from those fp16 values, in both places.
      uint16_t* wsT = ws + ((size_t)slot * Hv + h) * (2 * kWsTileElems);
      uint16_t* wsPT = wsT + kWsTileElems;
      for (int e = tid; e < kChunk * 8; e += kPrepThreads) {
        const int r = e >> 3, p = e & 7;
        uint4 v = *reinterpret_cast<const uint4*>(Th + r * LDB + 8 * p);
        uint32_t w4[4] = {v.x, v.y, v.z, v.w};
        if constexpr (F16) {
          *reinterpret_cast<uint4*>(Tmb + r * LDB + 8 * p) = v;
          const float dr = exp2f(g2[kChunk - 1] - g2[r]);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w4[q]));
            w4[q] = pack_f16(dr * f.x, dr * f.y);
          }
          *reinterpret_cast<uint4*>(wsT + r * kChunk + 8 * p) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
        } else {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w4[q]));
            w4[q] = pack16<false>(f.x, f.y);
          }
          v = make_uint4(w4[0], w4[1], w4[2], w4[3]);
          *reinterpret_cast<uint4*>(Tmb + r * LDB + 8 * p) = v;
          *reinterpret_cast<uint4*>(wsT + r * kChunk + 8 * p) = v;
        }
      }
      if (gi == G - 1) tc::fence_proxy_async();  // the inverse's working set is dead: the next tiles may land over it
      __syncthreads();
      if (gi == G - 1 && tid == 0) {  // the CTA's next item's tile copy overlaps PT and the stores
        for (int nx = item + (int)gridDim.x; nx < n_items; nx += gridDim.x) {
          Item it;
          if (locate(nx, it)) {
            load_tiles(nx, it);
            ahead = nx;
            break;
          }
        }
      }

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
                mma16<F16>(acc[2 * pp], a, bb[0], bb[1]);
                mma16<F16>(acc[2 * pp + 1], a, bb[2], bb[3]);
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
            *reinterpret_cast<uint32_t*>(Ps + r0 * LDB + cc) = pack16<F16>(acc[2 * pp + hh][0], acc[2 * pp + hh][1]);
            *reinterpret_cast<uint32_t*>(Ps + (r0 + 8) * LDB + cc) =
                pack16<F16>(acc[2 * pp + hh][2], acc[2 * pp + hh][3]);
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
// the array is malformed; every kernel clamps the entries to [0, T] all the same.  With
// `order`, it also writes the sequences most chunks first (chunk counts above 1022 share
// one bucket): the state carry dispatches its CTAs in that order, so that the longest chains
// do not start in the last wave.
__global__ void __launch_bounds__(1024)
gdn_chunk_table_kernel(const int32_t* __restrict__ cu, int B, int T, int32_t* __restrict__ chunk_off,
                       int32_t* __restrict__ order, int* __restrict__ err) {
  __shared__ int wsum[32];
  __shared__ int carry;
  __shared__ int bucket[1024];  // sequences per chunk count, most chunks first: key 1023 - min(chunks, 1023)
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

  // ---- dispatch order of the state carries: a counting sort on the chunk counts, most first
  // (sequences with the same count in any order; every sequence appears once) ----
  if (order == nullptr) return;
  auto key = [&](int b) {
    const int nc = (seq_bounds(cu, b, T).len + kChunk - 1) / kChunk;
    return 1023 - (nc < 1023 ? nc : 1023);
  };
  bucket[tid] = 0;
  __syncthreads();
  for (int b = tid; b < B; b += 1024) atomicAdd(&bucket[key(b)], 1);
  __syncthreads();
  // exclusive prefix sum of the 1024 bucket sizes (one per thread)
  {
    const int n = bucket[tid];
    int x = n;
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
      wsum[lane] = w;
    }
    __syncthreads();
    bucket[tid] = (warp ? wsum[warp - 1] : 0) + x - n;  // first position of the bucket
  }
  __syncthreads();
  for (int b = tid; b < B; b += 1024) order[atomicAdd(&bucket[key(b)], 1)] = b;
}

// ---- launchers -----------------------------------------------------------------
template <int DK, bool F16>
cudaError_t launch_prep_fmt(const CUtensorMap& mk, const CUtensorMap& mq, const float* g, const float* beta,
                            const int32_t* cu, const int32_t* chunk_off, void* ws, float* ws_rn, void* ws_kq, int* err,
                            int B, int T, int Hk, int Hv, int nslots, int nc_dense, int norm_qk, int hk_base,
                            int hk_count, int c_begin, int c_count, int persistent, cudaStream_t st) {
  using L = PrepSmem<DK>;
  cudaError_t e = set_smem_limit_once<gdn_prep_kernel<DK, F16>>(L::bytes);
  if (e != cudaSuccess) return e;
  if (cu == nullptr && (c_begin < 0 || c_count <= 0 || c_begin + c_count > nc_dense)) return cudaErrorInvalidValue;
  // items: key heads hk_base .. hk_base + hk_count - 1 of B sequences x c_count chunks (dense)
  // or of every slot (packed).  With the device to itself: persistent CTAs, as many per SM as fit.  Beside
  // other kernels (the host entry's pipelines) a CTA per item, so that the hardware spreads the
  // items over whatever SMs come free.
  const long long n_items = (cu == nullptr ? (long long)B * c_count : (long long)nslots) * hk_count;
  if (n_items <= 0) return cudaSuccess;
  if (n_items > 0x7fffffffLL) return cudaErrorInvalidValue;
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess ||
      (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
    return e;
  // kPrepCtasPerSm CTAs on every SM: the launch bounds keep the registers within an SM's
  // share, and all of the unified L1 / shared memory goes to shared memory (the driver's
  // default split fits fewer)
  static_assert(kPrepCtasPerSm * (L::bytes + 1024) <= 228 * 1024, "the CTAs of an SM do not fit in shared memory");
  static std::atomic<bool> carved[64] = {};
  if (dev < 0 || dev >= 64 || !carved[dev].load(std::memory_order_acquire)) {
    if ((e = cudaFuncSetAttribute(gdn_prep_kernel<DK, F16>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                  cudaSharedmemCarveoutMaxShared)) != cudaSuccess)
      return e;
    if (dev >= 0 && dev < 64) carved[dev].store(true, std::memory_order_release);
  }
  const long long resident = (long long)sms * kPrepCtasPerSm;
  const long long grid = persistent && n_items > resident ? resident : n_items;
  gdn_prep_kernel<DK, F16><<<(unsigned)grid, kPrepThreads, L::bytes, st>>>(
      mk, mq, g, beta, cu, chunk_off, static_cast<uint16_t*>(ws), ws_rn, static_cast<unsigned char*>(ws_kq), err, B,
      T, Hk, Hv, nc_dense, norm_qk, hk_base, hk_count, c_begin, c_count, (int)n_items);
  return cudaGetLastError();
}

// f16: the fp16 outputs (and [K; Q] image in ws_kq) of the default state carry; 0: bf16 tiles.
template <int DK>
cudaError_t launch_prep(const void* q, const void* k, const float* g, const float* beta,
                        const int32_t* cu, const int32_t* chunk_off, void* ws, float* ws_rn, void* ws_kq, int f16,
                        int* err, int B, int T, int Hk, int Hv, int nslots, int nc_dense, int norm_qk, int hk_base,
                        int hk_count, int c_begin, int c_count, int persistent, cudaStream_t st) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
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
  if (f16)
    return launch_prep_fmt<DK, true>(mk, mq, g, beta, cu, chunk_off, ws, ws_rn, ws_kq, err, B, T, Hk, Hv, nslots,
                                     nc_dense, norm_qk, hk_base, hk_count, c_begin, c_count, persistent, st);
  return launch_prep_fmt<DK, false>(mk, mq, g, beta, cu, chunk_off, ws, ws_rn, ws_kq, err, B, T, Hk, Hv, nslots,
                                    nc_dense, norm_qk, hk_base, hk_count, c_begin, c_count, persistent, st);
}

cudaError_t launch_chunk_table(const int32_t* cu, int B, int T, int32_t* chunk_off, int32_t* order, int* err,
                               cudaStream_t st) {
  gdn_chunk_table_kernel<<<1, 1024, 0, st>>>(cu, B, T, chunk_off, order, err);
  return cudaGetLastError();
}

#define GDN_INST_PREP(DK)                                                                                  \
  template cudaError_t launch_prep<DK>(const void*, const void*, const float*, const float*, const int32_t*, \
                                       const int32_t*, void*, float*, void*, int, int*, int, int, int, int, int, \
                                       int, int, int, int, int, int, int, cudaStream_t);
GDN_INST_PREP(32)
GDN_INST_PREP(64)
GDN_INST_PREP(128)

}  // namespace gdn
