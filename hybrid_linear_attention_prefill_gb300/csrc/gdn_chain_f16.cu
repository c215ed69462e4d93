// Chunk-sequential state carry with fp16 tensor-core operands: the library's default.
//
// It runs the chunk recurrence of the wide-range state carry (gdn_chain_tc.cu), one CTA per
// (sequence, value head, 16-, 32- or 64-row slice of S), 8 epilogue warps and 1 issue warp,
// the slice of S in fp32 registers.  With Tm = (I + A)^-1 and PT = P Tm from the preparation
// kernel, gamma = cumsum(g), e = exp(gamma), d = exp(gamma_last - gamma), the state update
// dS^T = K^T diag(d) U = K^T diag(d) Tm R associates as W R with
//
//   W = K^T diag(d) Tm        (dk x 64, no dependence on the state)
//
// so a chunk takes two dependent tensor-core rounds instead of three:
//
//   round 1   [X; Y] = [K; Q] S^T                       (M = 128 stacked tokens, K = dk)
//             R      = diag(beta) V - diag(beta e) X
//   round 2   dS^T   = W R                              (M = dk = 128, K = 64)
//             S      = e_last S + dS
//   beside    Z      = PT R, O = scale (diag(e) Y + Z)  -> bf16 outputs, during the next chunk
//   ahead     W of the next chunk = K^T (diag(d) Tm)    (M = 128, N = 64, K = 64), issued after
//             round 1; rounded to fp16 by the epilogue warps while the next chunk's round 1 runs
//
// the chunk form of S_t = a_t S_{t-1}(I - b_t k_t k_t^T) + b_t v_t k_t^T, o_t = S_t q_t / sqrt(dk)
// (the "chunked Gated DeltaNet prefill" of the "Open-Jev-27B-v1.1 native text worker" page,
// "Validation and optimization scope").  Z and W sit off the chain: only the R epilogue and
// the state update are between one chunk's round 1 and the next.
//
// Operands.  Every tensor-core operand is one fp16 value (kind::f16, fp32 accumulate): K and Q
// come from the preparation kernel as an fp16 image of the shared-memory tile, diag(d) Tm and PT
// are fp16 there as well, and W and the state-side operands S and R are rounded to fp16 from the
// fp32 values the epilogues hold.  fp16 keeps 11 significant bits where bf16 keeps 8, so a
// single fp16 operand replaces the bf16 hi + lo pair of the wide-range kernel: the MMAs carry
// N = DVT columns instead of 2 DVT, and the epilogues read and store half as many.  A float64
// model of the chunked path with these rounding points puts its errors below those of the bf16
// kernels (final state 4.3e-4 against 1.05e-3 relative, output 5.0e-4 against 2.5e-3 of the
// largest, on a no-decay, beta = 0.999 stress case): bf16 Tm was their largest rounding.
// fp16 stops at 65504.  An operand beyond it becomes infinite, and that reaches the state, so
// a (sequence, head) whose final fp32 state is not finite sets status bit 16 (also for
// non-finite inputs).  At the other end, fp16 keeps 11 bits only down to 2^-14; a state whose
// entries all stay below 2^-12 (values of order 1e-5 and less) has lost accuracy in its
// operands, so with check_small a CTA whose final state slice is nonzero but below 2^-12 sets
// status bit 32.  The wide-range kernel takes values of any magnitude.
//
// Shared-memory layouts (tile bases 1024-byte aligned):
//   [K; Q]    K-major, 128 B swizzle: [dk/64 blocks][128 rows][128 B]; rows 0..63 K, 64..127 Q
//             (the preparation kernel's image, one bulk copy per block).  The same K rows, read
//             MN-major (dk contiguous), are the A operand of the W product.
//   [dTm; PT] K-major, 128 B swizzle: [128 rows][128 B].  Rows 0..63 read MN-major (one 128-byte
//             row per token) are the B operand of the W product; rows 64..127 are Z's A operand
//             (the MMA's M = 128 rows start at row 0, and the Z rows 0..63 are not read).
//   S, R      MN-major, 128 B swizzle: one 128-byte row per K index (d or token), whose first
//             DVT fp16 values are the slice's columns (N = DVT of the row's 64).
//   V         the bf16 value slice: 32 B rows unswizzled (16 rows), 64 B rows with the 64 B
//             swizzle (32), 128 B rows with the 128 B swizzle (64).
// TMEM columns: round 1's [X; Y] in two buffers (the outputs read Y a chunk later), dS, Z, the
// fp32 W of the next chunk, and W in fp16 as dS's A operand (row d in lane d, two tokens a
// column) for this chunk and the next.  The epilogue warps round the next chunk's W while this
// chunk's dS is formed and write it with tcgen05.st: rounded into shared memory during round 1
// instead, it competed with round 1's operand reads and cost the headline step ~8 us.
#include <cuda_fp16.h>

#include "gdn_tc.cuh"
#include "gdn_tmap.cuh"

namespace gdn {

namespace {

constexpr int kThreads = 288;  // 8 epilogue warps + 1 issue warp
constexpr int kEpiThreads = 256;
constexpr uint32_t kMaxPolls = 1u << 24;
constexpr int kStatusNonFinite = 16;
constexpr int kStatusSmallState = 32;
constexpr float kSmallState = 1.f / 4096.f;  // 2^-12: two bits above fp16's smallest normal value

template <int DVT>
struct CfgH {
  static constexpr int kN = DVT;                 // MMA N: one fp16 column per state row
  static constexpr int kPS = kN < 32 ? 32 : kN;  // TMEM columns per accumulator
  static constexpr uint32_t kColD = 2 * kPS;     // dS (after the two [X; Y] buffers)
  static constexpr uint32_t kColZ = 3 * kPS;     // Z
  static constexpr uint32_t kColW = 4 * kPS;       // the next chunk's W, fp32 (64 columns)
  static constexpr uint32_t kColW16 = kColW + 64;  // W as dS's fp16 A operand, two chunks' (2 x 32 columns)
  static constexpr uint32_t kTmemCols = 4 * kPS + 128 <= 256 ? 256 : 512;
  static constexpr int kCPT = DVT / 2;                 // state columns per epilogue thread
  static constexpr int kGW = kCPT < 16 ? kCPT : 16;    // columns an epilogue step works on
  static constexpr int kNG = kCPT / kGW;               // steps per thread
  // stage layout (bytes)
  static constexpr int kOffKQ = 0;              // 2 x 16384
  static constexpr int kOffTP = 32768;          // 16384: [diag(d) Tm; PT]
  static constexpr int kOffV = kOffTP + 16384;  // 64 rows x 2 DVT bytes
  static constexpr int kVBytes = 64 * 2 * DVT;
  static constexpr int kOffG = kOffV + kVBytes;  // 64 fp32
  static constexpr int kOffB = kOffG + 256;      // 64 fp32
  static constexpr int kStage = (kOffB + 256 + 1023) / 1024 * 1024;  // 51, 53, 57 KB
  static constexpr int kStages = 3;  // chunk c + 2 loads during chunk c
  // after the stages: S (128 d rows) and R (64 token rows) as B operands, 128 B a row
  static constexpr int kOffS = kStages * kStage;
  static constexpr int kOffR = kOffS + 16384;
  static constexpr int kOffBar = kOffR + 8192;  // 5 MMA mbarriers, kStages load mbarriers, TMEM base, flags
  static constexpr int kSmemBytes = kOffBar + 128 + 1024;  // + slack for 1024-byte alignment
  static constexpr uint32_t kID_KS = tc::idesc_f16(128, kN, 0, 1);  // A K-major, B MN-major
  static constexpr uint32_t kID_W = tc::idesc_f16(128, 64, 1, 1);   // A MN-major, B MN-major
  static_assert(DVT == 16 || DVT == 32 || DVT == 64, "16, 32 or 64 state rows per CTA");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA");
  static_assert((5 + kStages) * 8 + 16 <= 128, "mbarriers and flags in the barrier block");
};

__device__ __forceinline__ uint32_t pack_h2(float a, float b) {
  __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

// W (8 or 16) consecutive fp32 columns of the warp's 32 TMEM lanes.
template <int W>
__device__ __forceinline__ void tmem_cols(uint32_t taddr, float (&acc)[W]) {
  static_assert(W == 8 || W == 16, "8 or 16 columns");
  if constexpr (W == 8) tc::tmem_ld8(taddr, acc);
  else tc::tmem_ld16(taddr, acc);
}

// W fp16 values at columns c0 .. c0 + W - 1 (c0 a multiple of 8) of operand row `row`:
// 16-byte chunks c0 / 8 .. of the 128-byte swizzled row.
template <int W>
__device__ __forceinline__ void store_h(unsigned char* tile, uint32_t row, int c0, const float* x) {
#pragma unroll
  for (int j = 0; j < W / 8; ++j)
    *reinterpret_cast<uint4*>(tile + tc::sw128(row, (uint32_t)(c0 / 8 + j))) =
        make_uint4(pack_h2(x[8 * j], x[8 * j + 1]), pack_h2(x[8 * j + 2], x[8 * j + 3]),
                   pack_h2(x[8 * j + 4], x[8 * j + 5]), pack_h2(x[8 * j + 6], x[8 * j + 7]));
}

// W bf16 values of token row `tok` of the value slice, columns c0 .. c0 + W - 1.
template <int DVT, int W>
__device__ __forceinline__ void load_v(const unsigned char* vt, int tok, int c0, float* vv) {
#pragma unroll
  for (int j = 0; j < W / 8; ++j) {
    const uint32_t ch = (uint32_t)(c0 / 8 + j);
    uint32_t off;
    if constexpr (DVT == 16) off = (uint32_t)tok * 32u + 16u * ch;
    else if constexpr (DVT == 32) off = tc::sw64((uint32_t)tok, ch);
    else off = tc::sw128((uint32_t)tok, ch);
    const uint4 raw = *reinterpret_cast<const uint4*>(vt + off);
    const uint32_t w4[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int p = 0; p < 4; ++p) {
      vv[8 * j + 2 * p] = __uint_as_float(w4[p] << 16);
      vv[8 * j + 2 * p + 1] = __uint_as_float(w4[p] & 0xffff0000u);
    }
  }
}

}  // namespace

// One CTA per SM.  Nine warps leave three on one of the SM's four sub-partitions, whose 16 K
// registers then cap a thread at 168.
template <int DK, int DVT>
__global__ void __launch_bounds__(kThreads, 1)
gdn_chain_f16_kernel(const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_w,
                     const unsigned char* __restrict__ ws_kq, const float* __restrict__ g,
                     const float* __restrict__ beta, const int32_t* __restrict__ cu,
                     const int32_t* __restrict__ chunk_off, const int32_t* __restrict__ order, const float* init,
                     __nv_bfloat16* __restrict__ out, float* fin, int* __restrict__ err, int B, int T, int Hk,
                     int Hv, int DV, int nc_dense, long long nslots, int h_base, int c_begin, int c_end,
                     int check_small) {
  // The value tiles are inputs, ready before the preparation kernel finishes: for dense batches
  // the issue thread brings the first chunks' tiles into L2 before the wait below.
  if (cu == nullptr && threadIdx.x == 256) {
    const int nt = DV / DVT;
    const int bb = (int)blockIdx.x / nt, d0 = ((int)blockIdx.x - bb * nt) * DVT, hh = h_base + (int)blockIdx.y;
    tc::prefetch_tensormap(&tm_v);
    for (int cc = c_begin; cc < c_begin + CfgH<DVT>::kStages && cc * kChunk < T; ++cc)
      tc::tma_prefetch_l2_3d(&tm_v, d0, hh, (int)((long long)bb * T + (long long)cc * kChunk));
  }
  using C = CfgH<DVT>;
  if (threadIdx.x == 0) {  // the barriers need nothing from the kernel before
    extern __shared__ unsigned char smem_raw[];
    const uint32_t r = smem_u32(smem_raw);
    uint64_t* bb = reinterpret_cast<uint64_t*>(smem_raw + (((r + 1023u) & ~1023u) - r) + C::kOffBar);
    for (int i = 0; i < 5 + C::kStages; ++i) tc::mbar_init(&bb[i], 1);
    tc::fence_mbar_init();
  }
  // Launched as a programmatic dependent of the kernel before it in the stream (the preparation
  // kernel): the CTA starts while that kernel's last CTAs run and waits here until it has
  // completed and its writes are visible (otherwise this returns at once).
  asm volatile("griddepcontrol.wait;\n" ::: "memory");
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw_s = smem_u32(smem_raw);
  const uint32_t pad = ((raw_s + 1023u) & ~1023u) - raw_s;
  unsigned char* sm = smem_raw + pad;
  const uint32_t sb = raw_s + pad;  // shared-window address of sm

  // [0] round 1, [1] dS, [2] Z: each completes once per chunk.  [3 + (j & 1)] the W of the
  // launch's chunk j.  W is issued before the barrier after which the epilogue warps wait for the
  // previous chunk's W, so one barrier could complete twice before a late warp polls it, and
  // its parity would then name a phase still to come; with two, the next completion of either
  // is issued only after every warp has passed the chunk's second barrier.
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + C::kOffBar);
  uint64_t* full = bars + 5;  // [0..kStages) stage loaded
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + C::kOffBar + 8 * (5 + C::kStages));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* state_max = reinterpret_cast<int*>(tmem_slot + 2);  // bits of the largest |S| (non-negative floats order as ints)

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const bool issuer = warp == 8;
  const int q4 = warp & 3;           // TMEM lane quadrant (epilogue warps)
  const int half = (warp >> 2) & 1;  // state columns kCPT half .. kCPT half + kCPT - 1
  const int row = 32 * q4 + lane;
  const int ntiles = DV / DVT;
  // CTA (x, y) = (sequence b x slices + slice, head).  With a dispatch order (packed batches),
  // the CTA's position in dispatch order walks the sequences most chunks first, and every
  // head and slice of one sequence before the next, so that the long chains start first.
  int bx = (int)blockIdx.x, hy = (int)blockIdx.y;
  if (order != nullptr) {
    const long long pos = (long long)blockIdx.y * gridDim.x + blockIdx.x;
    const int per = (int)gridDim.y * ntiles;  // CTAs of one sequence
    const int r = (int)(pos / per), rem = (int)(pos - (long long)r * per);
    const int ob = order[r];
    hy = rem / ntiles;
    bx = (ob >= 0 && ob < B ? ob : r) * ntiles + rem % ntiles;
  }
  const int b = bx / ntiles;
  const int dv0 = (bx - b * ntiles) * DVT;
  const int h = h_base + hy;
  const int hk = h / (Hv / Hk);
  const float scale = rsqrtf((float)DK);
  constexpr int kKBlocks = DK > 64 ? 2 : 1;  // 64-wide d blocks per tile
  constexpr uint32_t kTxBytes = kKBlocks * 16384 + C::kVBytes + 16384;
  constexpr int kAhead = C::kStages - 1;  // chunks whose tiles are in flight ahead of the current one
  constexpr int kCPT = C::kCPT, kGW = C::kGW, kNG = C::kNG;

  const SeqChunk sq = seq_bounds(cu, b, T);
  const int slot0 = cu == nullptr ? b * nc_dense : chunk_off[b];
  int nchunks = (sq.len + kChunk - 1) / kChunk;
  if ((long long)slot0 + nchunks > nslots) nchunks = slot0 < nslots ? (int)(nslots - slot0) : 0;
  // this launch walks chunks c0 .. c1 - 1 of the sequence, from `init` (the state before
  // chunk c0) to `fin` (the state after chunk c1 - 1)
  const int c0 = c_begin < nchunks ? c_begin : nchunks;
  const int c1 = c_end < nchunks ? c_end : nchunks;

  // ---- set-up: TMEM, barriers, zero d-block 1 when dk <= 64 --------------------
  if (warp == 0) {
    tc::tmem_alloc(tmem_slot, C::kTmemCols);
    tc::tmem_relinquish();
  }
  if (tid == 0) {
    *abort_flag = 0;
    *state_max = 0;
    tc::fence_mbar_init();
  }
  if (issuer && lane == 0) {
    tc::prefetch_tensormap(&tm_v);
    tc::prefetch_tensormap(&tm_w);
  }
  if (kKBlocks == 1 && !issuer) {  // the W product reads all 128 rows of K^T: the rows d >= 64 stay zero
    for (int e = tid; e < C::kStages * 1024; e += kEpiThreads) {
      const int stg = e >> 10, w = e & 1023;
      *reinterpret_cast<uint4*>(sm + stg * C::kStage + C::kOffKQ + 16384 + w * 16) = make_uint4(0, 0, 0, 0);
    }
  }

  // ---- initial state: thread (row d, half) holds S[kCPT half + i][d] ----------------
  const int d = row;
  float s[kCPT];
  if (!issuer) {
    const size_t base = ((size_t)b * Hv + h) * DV + dv0 + kCPT * half;
#pragma unroll
    for (int i = 0; i < kCPT; ++i) s[i] = (init != nullptr && d < DK) ? init[(base + i) * DK + d] : 0.f;
#pragma unroll
    for (int gg = 0; gg < kNG; ++gg) store_h<kGW>(sm + C::kOffS, d, kCPT * half + kGW * gg, s + kGW * gg);
  }
  tc::fence_proxy_async();
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tq = tmem + ((uint32_t)(32 * q4) << 16);  // this warp's lanes

  // bulk copies and TMA for the tiles of chunk c into stage stg (one thread); g and beta by cp.async.
  auto load_tiles = [&](int c, int stg) {
    unsigned char* st = sm + stg * C::kStage;
    const int t0 = (int)(sq.bos + (long long)c * kChunk);
    const unsigned char* kq = ws_kq + ((size_t)(slot0 + c) * Hk + hk) * kws_kq_bytes(DK);
    tc::mbar_arrive_expect_tx(&full[stg], kTxBytes);
#pragma unroll
    for (int db = 0; db < kKBlocks; ++db) tc::bulk_load(st + C::kOffKQ + db * 16384, kq + db * 16384, 16384, &full[stg]);
    tc::tma_load_2d(st + C::kOffTP, &tm_w, 0, (int)(((long long)(slot0 + c) * Hv + h) * 128), &full[stg]);
    tc::tma_load_3d(st + C::kOffV, &tm_v, dv0, h, t0, &full[stg]);
  };
  auto load_scalars = [&](int c, int stg) {
    unsigned char* st = sm + stg * C::kStage;
    if (tid < kChunk) {
      const int n = min(kChunk, sq.len - c * kChunk);
      const bool ok = tid < n;
      const size_t off = ok ? (size_t)(sq.bos + (long long)c * kChunk + tid) * Hv + h : 0;
      cp_async4(st + C::kOffG + 4 * tid, g + off, ok);
      cp_async4(st + C::kOffB + 4 * tid, beta + off, ok);
    }
  };
  // W = K^T (diag(d) Tm) of the chunk in stage stg: A the K rows read MN-major, B the diag(d) Tm
  // rows read MN-major (one 128-byte row per token), fp32 into TMEM columns kColW .. + 63.
  auto issue_w = [&](int stg, int wb) {  // wb: the chunk's position in the launch, mod 2
    const uint32_t base = sb + (uint32_t)(stg * C::kStage);
    const uint64_t ka = tc::sdesc(base + C::kOffKQ, 16384, 1024, tc::kSw128);
    const uint64_t tb = tc::sdesc(base + C::kOffTP, 8192, 1024, tc::kSw128);
#pragma unroll
    for (int ks = 0; ks < 4; ++ks)
      tc::mma_bf16(tmem + C::kColW, ka + (uint64_t)((ks * 2048) >> 4), tb + (uint64_t)((ks * 2048) >> 4), C::kID_W,
                   ks > 0);
    tc::commit(&bars[3 + wb]);
  };
  // The W of the launch's chunk j to fp16 (epilogue warps): rows d = 32 q4 + lane, tokens
  // 32 half .. + 31, into the chunk's W buffer in TMEM.  The stores are complete when it returns.
  auto convert_w = [&](int j) {
    if (!tc::mbar_wait(&bars[3 + (j & 1)], (uint32_t)((j >> 1) & 1), kMaxPolls)) {
      *abort_flag = 1;
      atomicOr(err, 1);
    }
    tc::fence_after();
    float w0[16], w1[16];
    tc::tmem_ld16(tq + C::kColW + 32 * half, w0);
    tc::tmem_ld16(tq + C::kColW + 32 * half + 16, w1);
    uint32_t h16[16];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      h16[i] = pack_h2(w0[2 * i], w0[2 * i + 1]);
      h16[8 + i] = pack_h2(w1[2 * i], w1[2 * i + 1]);
    }
    tc::tmem_st16(tq + C::kColW16 + 32 * (j & 1) + 16 * half, h16);
  };

  if (c1 > c0) {
    if (issuer && lane == 0) {
      for (int a = 0; a < kAhead && c0 + a < c1; ++a) load_tiles(c0 + a, a);
      // the first chunk's W (the later ones are formed a chunk ahead)
      if (!tc::mbar_wait(&full[0], 0u, kMaxPolls)) {
        *abort_flag = 1;
        atomicOr(err, 2);
      } else {
        issue_w(0, 0);
      }
    }
    load_scalars(c0, 0);
  }
  cp_async_commit();
  // the first chunk's W to fp16 (the later ones are rounded a chunk ahead, while the chunk
  // before forms its dS), before the issuing thread reuses the fp32 W columns
  __syncthreads();
  if (c1 > c0 && !issuer && !*abort_flag) convert_w(0);
  tc::fence_before();

  const int tok = 32 * (q4 & 1) + lane;  // this thread's token in the R and output epilogues
  // shared-memory descriptors of the operands at stage 0 / their buffers (the issuer's MMAs)
  const uint64_t dKQ0 = tc::sdesc(sb + C::kOffKQ, 16, 1024, tc::kSw128);  // [K; Q], K-major
  const uint64_t dTP0 = tc::sdesc(sb + C::kOffTP, 16, 1024, tc::kSw128);  // [dTm; PT], K-major
  const uint64_t dS = tc::sdesc(sb + C::kOffS, 16384, 1024, tc::kSw128);  // S, MN-major
  const uint64_t dR = tc::sdesc(sb + C::kOffR, 8192, 1024, tc::kSw128);   // R, MN-major
  // the outputs of the chunk before: its e, token count and output row
  float e_prev = 0.f;
  int n_prev = 0;
  __nv_bfloat16* orow_prev = out;
  bool aborted = false;
  int c = c0;
  for (; c < c1; ++c) {
    const int ci = c - c0;  // position in this launch: stage and barrier phases
    const int stg = ci % C::kStages;
    const uint32_t par = (uint32_t)(ci & 1);
    const uint32_t col1 = (uint32_t)C::kPS * par;  // this chunk's [X; Y] buffer
    unsigned char* st = sm + stg * C::kStage;
    cp_async_wait<0>();
    // The stage's tiles: the issuing thread waited for them before forming this chunk's W (a
    // chunk earlier), and the barrier below publishes them to every thread (it makes the
    // accesses that thread requested and saw complete visible to all the CTA's threads).
    __syncthreads();
    // Every thread reads the abort flag right after each barrier, so all of them leave the loop
    // at the same barrier; the issuing thread acts on it after issuing that round's MMAs (which
    // an abort makes harmless), so the read is off its path to the tensor core.
    const int ab_top = *abort_flag;

    if (issuer) {
      // Descriptors: this stage's bases plus each MMA's offset, added to the start-address field
      // (byte offset / 16; shared addresses stay below 2^18, so the 14-bit field does not carry).
      const uint64_t dKQ = dKQ0 + (uint64_t)((uint32_t)(stg * C::kStage) >> 4);
      const uint64_t dTP = dTP0 + (uint64_t)((uint32_t)(stg * C::kStage) >> 4);
      // ---- round 1: [X; Y] = [K; Q] S^T ---------------------------------------------
      if (lane == 0) {
        tc::fence_after();
#pragma unroll
        for (int ks = 0; ks < DK / 16; ++ks) {
          const uint64_t a = dKQ + (uint64_t)(((ks >> 2) * 16384 + (ks & 3) * 32) >> 4);
          const uint64_t bd = dS + (uint64_t)((ks * 2048) >> 4);
          tc::mma_bf16(tmem + col1, a, bd, C::kID_KS, ks > 0);
        }
        tc::commit(&bars[0]);
        // the next chunk's W, once its tiles are in (rounded to fp16 while this chunk's dS runs)
        if (c + 1 < c1) {
          const int s1 = (ci + 1) % C::kStages;
          if (!tc::mbar_wait(&full[s1], (uint32_t)(((ci + 1) / C::kStages) & 1), kMaxPolls)) {
            *abort_flag = 1;
            atomicOr(err, 2);
          } else {
            issue_w(s1, (ci + 1) & 1);
          }
        }
      }
      __syncwarp();
      if (ab_top) { aborted = true; break; }
      __syncthreads();  // R written
      const int ab_r = *abort_flag;
      // ---- round 2: dS^T = W R; then Z = PT R, off the chain -------------------------
      if (lane == 0) {
        tc::fence_after();
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          tc::mma_f16_ta(tmem + C::kColD, tmem + C::kColW16 + 32 * par + 8 * ks, dR + (uint64_t)((ks * 2048) >> 4),
                         C::kID_KS, ks > 0);
        tc::commit(&bars[1]);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          tc::mma_bf16(tmem + C::kColZ, dTP + (uint64_t)((ks * 32) >> 4), dR + (uint64_t)((ks * 2048) >> 4), C::kID_KS,
                       ks > 0);
        tc::commit(&bars[2]);
      }
      __syncwarp();
      if (ab_r) { aborted = true; break; }
      continue;
    }

    // ================= epilogue warps =================
    if (ab_top) { aborted = true; break; }
    if (c + 1 < c1) load_scalars(c + 1, (ci + 1) % C::kStages);
    cp_async_commit();

    // per-token scalars: every warp scans the 64 log decays of the chunk
    const float* gs = reinterpret_cast<const float*>(st + C::kOffG);
    const float* bs = reinterpret_cast<const float*>(st + C::kOffB);
    float g0 = gs[lane], g1 = gs[lane + 32];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float u0 = __shfl_up_sync(0xffffffffu, g0, o);
      const float u1 = __shfl_up_sync(0xffffffffu, g1, o);
      if (lane >= o) { g0 += u0; g1 += u1; }
    }
    g1 += __shfl_sync(0xffffffffu, g0, 31);
    const float glast = __shfl_sync(0xffffffffu, g1, 31);
    const float gam = (q4 & 1) ? g1 : g0;
    const float e_t = expf(gam);
    const float eC = expf(glast);

    if (q4 < 2) {
      // ---- R = beta V - beta e X (rows 0..63 of round 1) ----------------------------------
      const float b_t = bs[tok];
      if (!tc::mbar_wait(&bars[0], par, kMaxPolls)) { *abort_flag = 1; atomicOr(err, 1); }
      tc::fence_after();
#pragma unroll
      for (int gg = 0; gg < kNG; ++gg) {
        const int cc = kCPT * half + kGW * gg;  // slice column of this step
        float acc[kGW];
        tmem_cols<kGW>(tq + col1 + cc, acc);
        float vv[kGW];
        load_v<DVT, kGW>(st + C::kOffV, tok, cc, vv);
        const float be = b_t * e_t;
#pragma unroll
        for (int i = 0; i < kGW; ++i) acc[i] = b_t * vv[i] - be * acc[i];
        store_h<kGW>(sm + C::kOffR, tok, cc, acc);
      }
    } else {
      // ---- the previous chunk's outputs from its Y (rows 64..127 of its round 1) and Z ----
      if (ci > 0) {
        if (!tc::mbar_wait(&bars[2], par ^ 1u, kMaxPolls)) { *abort_flag = 1; atomicOr(err, 1); }
        tc::fence_after();
      }
      // The stage of the previous chunk is free once its Z is done: its tiles for chunk c + 2.
      if (warp == 2 && lane == 0 && c + kAhead < c1) load_tiles(c + kAhead, (ci + kAhead) % C::kStages);
      if (ci > 0) {
        const uint32_t colp = (uint32_t)C::kPS * (par ^ 1u);
        const float es = scale * e_prev;
#pragma unroll
        for (int gg = 0; gg < kNG; ++gg) {
          const int cc = kCPT * half + kGW * gg;
          float y[kGW], z[kGW];
          tmem_cols<kGW>(tq + colp + cc, y);
          tmem_cols<kGW>(tq + C::kColZ + cc, z);
          if (tok < n_prev) {
#pragma unroll
            for (int j = 0; j < kGW / 8; ++j) {
              uint32_t o4[4];
#pragma unroll
              for (int p = 0; p < 4; ++p)
                o4[p] = pack_bf16(es * y[8 * j + 2 * p] + scale * z[8 * j + 2 * p],
                                  es * y[8 * j + 2 * p + 1] + scale * z[8 * j + 2 * p + 1]);
              *reinterpret_cast<uint4*>(orow_prev + cc + 8 * j) = make_uint4(o4[0], o4[1], o4[2], o4[3]);
            }
          }
        }
      }
    }
    if (q4 < 2) tc::fence_proxy_async();  // R is read by the tensor core next
    tc::fence_before();
    __syncthreads();  // R written
    if (*abort_flag) { aborted = true; break; }

    // the next chunk's W (issued after this chunk's round 1) to fp16 while dS is formed
    if (c + 1 < c1) convert_w(ci + 1);

    // ---- S = e_last S + dS ------------------------------------------------------------
    if (!tc::mbar_wait(&bars[1], par, kMaxPolls)) { *abort_flag = 1; atomicOr(err, 1); }
    tc::fence_after();
#pragma unroll
    for (int gg = 0; gg < kNG; ++gg) {
      const int cc = kCPT * half + kGW * gg;
      float acc[kGW];
      tmem_cols<kGW>(tq + C::kColD + cc, acc);
#pragma unroll
      for (int i = 0; i < kGW; ++i) s[kGW * gg + i] = fmaf(eC, s[kGW * gg + i], acc[i]);
      store_h<kGW>(sm + C::kOffS, d, cc, s + kGW * gg);
    }
    tc::fence_proxy_async();  // S is read by the tensor core at the next chunk
    tc::fence_before();
    e_prev = e_t;
    n_prev = min(kChunk, sq.len - c * kChunk);
    orow_prev = out + ((size_t)(sq.bos + (long long)c * kChunk + tok) * Hv + h) * DV + dv0;
  }

  // ---- the last chunk's outputs, final state, clean-up ------------------------------------
  cp_async_wait<0>();
  if (!aborted && !issuer && q4 >= 2 && c1 > c0) {
    const uint32_t pl = (uint32_t)((c1 - 1 - c0) & 1);
    if (tc::mbar_wait(&bars[2], pl, kMaxPolls)) {
      tc::fence_after();
      const float es = scale * e_prev;
#pragma unroll
      for (int gg = 0; gg < kNG; ++gg) {
        const int cc = kCPT * half + kGW * gg;
        float y[kGW], z[kGW];
        tmem_cols<kGW>(tq + (uint32_t)C::kPS * pl + cc, y);
        tmem_cols<kGW>(tq + C::kColZ + cc, z);
        if (tok < n_prev) {
#pragma unroll
          for (int j = 0; j < kGW / 8; ++j) {
            uint32_t o4[4];
#pragma unroll
            for (int p = 0; p < 4; ++p)
              o4[p] = pack_bf16(es * y[8 * j + 2 * p] + scale * z[8 * j + 2 * p],
                                es * y[8 * j + 2 * p + 1] + scale * z[8 * j + 2 * p + 1]);
            *reinterpret_cast<uint4*>(orow_prev + cc + 8 * j) = make_uint4(o4[0], o4[1], o4[2], o4[3]);
          }
        }
      }
    } else {
      atomicOr(err, 1);
    }
  }
  if (!aborted && !issuer && d < DK) {
    bool finite = true;
    float mx = 0.f;
#pragma unroll
    for (int i = 0; i < kCPT; ++i) {
      finite = finite && fabsf(s[i]) <= 3.402823466e38f;
      mx = fmaxf(mx, fabsf(s[i]));
    }
    if (!finite) atomicOr(err, kStatusNonFinite);
    if (check_small) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(__activemask(), mx, o));
      if (lane == 0) atomicMax(state_max, __float_as_int(mx));
    }
    if (fin != nullptr) {
      const size_t base = ((size_t)b * Hv + h) * DV + dv0 + kCPT * half;
#pragma unroll
      for (int i = 0; i < kCPT; ++i) fin[(base + i) * DK + d] = s[i];
    }
  }
  if (aborted && issuer && lane == 0) {
    // let MMAs and copies still in flight land before the CTA exits (bounded again; a phase
    // that never started just runs out of polls)
    for (int i = 0; i < 5; ++i)
      for (uint32_t p = 0; p < 2; ++p) (void)tc::mbar_wait(&bars[i], p, 1u << 14);
    for (int i = 0; i < C::kStages; ++i)
      for (uint32_t p = 0; p < 2; ++p) (void)tc::mbar_wait(&full[i], p, 1u << 14);
  }
  tc::fence_before();
  __syncthreads();
  if (check_small && !aborted && tid == 0) {
    const float mx = __int_as_float(*state_max);
    if (mx > 0.f && mx < kSmallState) atomicOr(err, kStatusSmallState);
  }
  if (warp == 0) tc::tmem_dealloc(tmem, C::kTmemCols);
}

template <int DK, int DVT>
cudaError_t launch_chain_f16_dvt(const void* v, const CUtensorMap& mw, const void* ws_kq, const float* g,
                                 const float* beta, const int32_t* cu, const int32_t* chunk_off,
                                 const int32_t* order, const float* init, void* out, float* fin, int* err, int B,
                                 int T, int Hk, int Hv, int DV, int nc_dense, long long nslots, int h_base,
                                 int h_count, int c_begin, int c_end, int check_small, cuuint64_t tt,
                                 cudaStream_t st) {
  using C = CfgH<DVT>;
  CUtensorMap mv;
  {
    const cuuint64_t dims[3] = {(cuuint64_t)DV, (cuuint64_t)Hv, tt};
    const cuuint64_t strides[2] = {(cuuint64_t)DV * 2, (cuuint64_t)Hv * DV * 2};
    const cuuint32_t box[3] = {DVT, 1, 64};
    const CUtensorMapSwizzle swz =
        DVT == 16 ? CU_TENSOR_MAP_SWIZZLE_NONE : DVT == 32 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B;
    if (!make_map16(&mv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, v, 3, dims, strides, box, swz))
      return cudaErrorInvalidValue;
  }
  cudaError_t e = set_smem_limit_once<gdn_chain_f16_kernel<DK, DVT>>(C::kSmemBytes);
  if (e != cudaSuccess) return e;
  // value heads h_base .. h_base + h_count - 1; a programmatic dependent of the kernel before it
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)B * (DV / DVT), h_count);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, gdn_chain_f16_kernel<DK, DVT>, mv, mw, static_cast<const unsigned char*>(ws_kq), g,
                         beta, cu, chunk_off, order, init, static_cast<__nv_bfloat16*>(out), fin, err, B, T, Hk,
                         Hv, DV, nc_dense, nslots, h_base, c_begin, c_end, check_small);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// check_small: report a final state below fp16's accurate range (status bit 32); off for the
// two-level scan's inner runs, whose transition states may be legitimately tiny.
// slice: state rows per CTA, 16, 32 or 64, or 0 for the library's choice.  The MMA issue and
// the hand-offs of a chunk step do not depend on the width and its epilogues scale with it:
// measured at 64 chunks (state carry alone), a 16-row step takes 0.97-1.0x a 32-row one and a
// 64-row step 1.19x.  So 64 rows when dv allows it and 1.19 x its waves of one CTA per SM are
// fewer than the 32-row grid's waves (many sequences or heads); 16 rows when twice the 32-row
// grid still fits one wave (few heads: the chain latency decides, and narrower slices shorten it
// a little); 32 otherwise.
template <int DK>
cudaError_t launch_chain_f16(const void* v, const float* g, const float* beta, const int32_t* cu,
                             const int32_t* chunk_off, const int32_t* order, const void* ws, const void* ws_kq,
                             const float* init, void* out, float* fin, int* err, int B, int T, int Hk, int Hv,
                             int DV, int nc_dense, long long nslots, int h_base, int h_count, int c_begin,
                             int c_end, int slice, int check_small, cudaStream_t st) {
  const long long ttot = cu != nullptr ? (long long)T : (long long)B * T;
  const cuuint64_t tt = (cuuint64_t)(ttot > 0 ? ttot : 1);
  CUtensorMap mw;
  {
    const long long rows = nslots * Hv * 128;
    const cuuint64_t dims[2] = {64, (cuuint64_t)(rows > 0 ? rows : 1)};
    const cuuint64_t strides[1] = {128};
    const cuuint32_t box[2] = {64, 128};
    if (!make_map16(&mw, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, ws, 2, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  }
  if (slice == 0) {
    slice = 32;
    int dev = 0, sms = 0;
    cudaError_t e;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return e;
    const long long n32 = (long long)B * (DV / 32) * h_count;
    const long long waves32 = (n32 + sms - 1) / sms, waves64 = (n32 / 2 + sms - 1) / sms;
    if (DV % 64 == 0 && 119 * waves64 < 100 * waves32) slice = 64;
    else if (2 * n32 <= sms) slice = 16;
  }
  switch (slice) {
    case 16:
      return launch_chain_f16_dvt<DK, 16>(v, mw, ws_kq, g, beta, cu, chunk_off, order, init, out, fin, err, B, T, Hk,
                                          Hv, DV, nc_dense, nslots, h_base, h_count, c_begin, c_end, check_small,
                                          tt, st);
    case 32:
      return launch_chain_f16_dvt<DK, 32>(v, mw, ws_kq, g, beta, cu, chunk_off, order, init, out, fin, err, B, T, Hk,
                                          Hv, DV, nc_dense, nslots, h_base, h_count, c_begin, c_end, check_small,
                                          tt, st);
    case 64:
      if (DV % 64 != 0) return cudaErrorInvalidValue;
      return launch_chain_f16_dvt<DK, 64>(v, mw, ws_kq, g, beta, cu, chunk_off, order, init, out, fin, err, B, T, Hk,
                                          Hv, DV, nc_dense, nslots, h_base, h_count, c_begin, c_end, check_small,
                                          tt, st);
    default:
      return cudaErrorInvalidValue;
  }
}

#define GDN_INST_CHAIN_F16(DK)                                                                                 \
  template cudaError_t launch_chain_f16<DK>(const void*, const float*, const float*, const int32_t*,           \
                                            const int32_t*, const int32_t*, const void*, const void*,          \
                                            const float*, void*, float*, int*, int, int, int, int, int, int,   \
                                            long long, int, int, int, int, int, int, cudaStream_t);
GDN_INST_CHAIN_F16(32)
GDN_INST_CHAIN_F16(64)
GDN_INST_CHAIN_F16(128)

}  // namespace gdn
