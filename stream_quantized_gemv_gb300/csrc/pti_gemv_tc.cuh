// pti_gemv_tc.cuh -- the tensor-core consumer of the Q8 GEMV kernel.
//
// Included by pti_gemv_kernel.cuh inside its namespace: it reuses the stage
// ring and its copy producer, the tile finishing, the tile-combine kernel and
// the fused epilogues defined there, and replaces only the consumer side.
// Launches select it with PTI_FLAG_TENSOR_CORES; the CUDA-core consumer is
// the default, because this one measured no faster (see the end of this
// comment).
//
// Aim: one weight load serves N activation streams ([PTI-readme]
// "打包双子推理（PTI）" §"带宽分析：为什么会有开销"), but on the CUDA cores each
// weight then costs 1 + N fp32 FMA lane-operations (the exact q d and one
// product per stream) and a byte permute, which at N = 4 is more than the
// FP32 pipe retires while HBM delivers the weights.  Here the per-stream
// products run on the tensor core, and the CUDA cores only convert:
//
//  * A (tensor memory, binary16): every int8 weight q is exactly a binary16
//    value.  A converter thread owns one row of the 128-row unit and four of
//    its eight blocks; it turns each block's 32 bytes into 16 f16x2 words (a
//    byte permute into the binary16 pattern of 1024 + (q + 128), then one
//    packed add of -1152, both exact) and writes them with tcgen05.st into the
//    row's tensor-memory lane.  The block's scale d stays in a register.
//  * B (shared memory, binary16): the activations of stream n are scaled by a
//    power of two 2^k, chosen per (block, stream) so that the block's largest
//    |x| lies in [2^14, 2^15), and each x 2^k is split into three binary16
//    pieces h + m + l (h = x 2^k rounded to binary16, m = the remainder
//    rounded, l = what is left).  With 11 significant bits each, the pieces
//    hold all 24 bits of the fp32 value, except for elements 2^15 or more
//    below their block's largest, whose error stays below 2^-39 of that
//    largest.  The pieces of stream n are rows 3n, 3n + 1, 3n + 2 of the
//    unit's 16-row B (unused rows zero), K-major without swizzle.
//  * One tcgen05.mma (M = 128, N = 16, K = 16, fp32 accumulation) per half
//    block: each of the block's 32 products q x_piece is exact in fp32 and
//    the tensor core sums them.  Blocks do not share an accumulator (every row
//    has its own scale per block): the unit's 8 blocks fill 8 x 16 columns of
//    D.
//  * One unit behind the conversion (so that the tensor core's latency hides
//    behind the next unit's conversion) the converter threads load their
//    row's D columns with tcgen05.ld and add, per block and stream,
//    ((h + (m + l)) d) 2^-k to the row's unit sum, which goes to the row's
//    accumulator once per unit, as on the CUDA-core path.
//
// Tensor memory: 512 columns, A and D of two units in flight (128 columns
// each).  Warps 0..7 convert (warp w: rows 32 (w % 4) .. +31 -- the lanes a
// warp may access -- and blocks 4 (w / 4) .. +3; for the activation pieces,
// block w), warp 8 issues the copies (the CUDA-core kernel's producer), lane
// 0 of warp 9 issues the MMAs and owns the tensor-memory allocation.
//
// Measured on GB300 (17408 x 5120, four streams, chained launches): about
// 28.2 us per GEMV against 28.8 us for the CUDA-core consumer; this one is
// bound by the tensor core's instruction rate, that one by its FMA pipe,
// neither by HBM.  K = 16 per
// kind::f16 instruction makes 16 MMAs per 128 x 256 unit; alone, one such MMA
// (N <= 64) occupies the tensor pipe about 47 SM cycles whatever N, but with
// the conversion's shared- and tensor-memory traffic running beside it, each
// took 170-200 cycles, so 16 of them cost about as long as the CUDA cores'
// 1 + N FMAs per weight.  (Sixteen converter warps, one tcgen05.st of 32
// columns instead of two of 16, and paired activation stores each measured
// slower: they only add to that traffic.)

constexpr int kTcWarps = 8;                        // converter warps
constexpr int kTcThreads = kTcWarps * 32;
constexpr int kTcBBytes = 16 * 256 * 2;            // one unit's B: 16 rows x 256 columns of binary16
constexpr uint32_t kTcCols = 512;                  // tensor-memory columns: A[2], D[2]
constexpr uint32_t kTcAOff = 0, kTcDOff = 256;     // first column of A[0] and of D[0]
constexpr uint32_t kBarTcExit = 2;                 // named barrier: converter warps and the MMA warp
// Instruction descriptor of tcgen05.mma kind::f16: D fp32 (bits 4-5 = 1),
// A and B binary16 (bits 7-9, 10-12 = 0), both K-major (bits 15, 16 = 0),
// N / 8 in bits 17-22, M / 16 in bits 24-28.
constexpr uint32_t kTcIdesc = (1u << 4) | ((16u >> 3) << 17) | ((128u >> 4) << 24);
constexpr uint32_t kTcLbo = 256;  // B: bytes between core matrices adjacent in K (8 columns)
constexpr uint32_t kTcSbo = 128;  // B: bytes between core matrices adjacent in N (8 rows)

// Byte offset of B element (row, column) in the unit's B: 8 x 8 core
// matrices of 128 bytes (8 rows of 16 bytes), the two row groups of a column
// group next to each other.
__device__ __forceinline__ uint32_t tc_b_offset(uint32_t row, uint32_t col) {
  return (col >> 3) * kTcLbo + (row >> 3) * kTcSbo + (row & 7u) * 16u + (col & 7u) * 2u;
}

// Shared-memory matrix descriptor of a K-major, unswizzled operand starting at
// shared address `saddr` (16-byte aligned): start >> 4 in bits 0-13, the K
// stride >> 4 in bits 16-29, the N stride >> 4 in bits 32-45, descriptor
// version 1 in bits 46-47, no swizzle (bits 61-63 = 0).
__device__ __forceinline__ uint64_t tc_smem_desc(uint32_t saddr) {
  return static_cast<uint64_t>((saddr >> 4) & 0x3FFFu) | (static_cast<uint64_t>(kTcLbo >> 4) << 16) |
         (static_cast<uint64_t>(kTcSbo >> 4) << 32) | (1ull << 46);
}

template <int N>
struct TcLayout {
  static constexpr int kXinvBytes = 3 * 8 * 4 * 4;              // [unit % 3][block][stream] 2^-k
  static constexpr int kRedBytes = 2 * 2 * N * kRowsPerTile * 4;  // [slot][block group][stream][row]
};

// Totals policy: two parked sums per element (block groups 0-3 and 4-7).
template <int N>
struct TcTotals {
  static constexpr int kThreads = kTcThreads;
  template <int kOut>
  __device__ __forceinline__ static float total(const float *red, int sl, int s, int row) {
    return red[((sl * 2 + 0) * kOut + s) * kRowsPerTile + row] + red[((sl * 2 + 1) * kOut + s) * kRowsPerTile + row];
  }
};

// The activation pieces of one unit: warp w handles block w, lane l its
// column 32 w + l, for every stream.  Writes B and the block's 2^-k per
// stream (lane 0).
template <int N>
__device__ __forceinline__ void tc_split_x(const float *xs, uint8_t *bop, float *xinv, uint32_t warp,
                                           uint32_t lane) {
  const uint32_t col = 32u * warp + lane;
#pragma unroll
  for (int n = 0; n < N; ++n) {
    const float x = xs[n * 256 + col];
    // biased exponent of the block's largest |x| (0 for zeros and subnormals)
    const uint32_t e = __reduce_max_sync(0xFFFFFFFFu, __float_as_uint(x) & 0x7F800000u) >> 23;
    const int k = min(141 - static_cast<int>(e), 126);  // largest |x| 2^k in [2^14, 2^15); 2^k, 2^-k normal
    const float xp = x * __uint_as_float(static_cast<uint32_t>(k + 127) << 23);
    const uint32_t h = float_to_half_bits(xp);
    const float r1 = xp - half_bits_to_float(h);  // exact
    const uint32_t m = float_to_half_bits(r1);
    const float r2 = r1 - half_bits_to_float(m);  // exact
    const uint32_t l = float_to_half_bits(r2);
    *reinterpret_cast<uint16_t *>(bop + tc_b_offset(3u * n, col)) = static_cast<uint16_t>(h);
    *reinterpret_cast<uint16_t *>(bop + tc_b_offset(3u * n + 1u, col)) = static_cast<uint16_t>(m);
    *reinterpret_cast<uint16_t *>(bop + tc_b_offset(3u * n + 2u, col)) = static_cast<uint16_t>(l);
    if (lane == 0) xinv[warp * 4 + n] = __uint_as_float(static_cast<uint32_t>(127 - k) << 23);
  }
}

// Converts blocks 4G .. 4G+3 of one row of a unit (row pointer `rowp` into
// the stage's weight tile) into tensor memory at column `ta` + 16 b for block
// b, and returns the blocks' scales.  The four blocks are bytes 136 G ..
// 136 G + 135 of the 272-byte row: nine aligned 16-byte loads from byte
// 128 G.  Block 4G + t starts at byte off = 34 t + 8 G of that window: its
// scale is half-word off % 4 / 2 of word off / 4, weight pair i (columns 2i,
// 2i + 1) is at byte off + 2 + 2i, which is 0 or 2 mod 4, so both weights
// of a pair sit in one aligned word.
template <int G>
__device__ __forceinline__ void tc_convert(const uint8_t *rowp, uint32_t ta, float (&d)[4]) {
  uint32_t w[36];
#pragma unroll
  for (int k = 0; k < 9; ++k) {
    const uint4 v = *reinterpret_cast<const uint4 *>(rowp + 128 * G + 16 * k);
    w[4 * k] = v.x;
    w[4 * k + 1] = v.y;
    w[4 * k + 2] = v.z;
    w[4 * k + 3] = v.w;
  }
  static_for<0, 4>([&](auto t_) {
    constexpr int t = decltype(t_)::value;
    constexpr int off = 34 * t + 8 * G;
    d[t] = half_bits_to_float(off % 4 == 0 ? (w[off / 4] & 0xFFFFu) : (w[off / 4] >> 16));
    uint32_t o[16];
    static_for<0, 16>([&](auto i_) {
      constexpr int i = decltype(i_)::value;
      constexpr int p = off + 2 + 2 * i;
      // bytes [u_2i, 0x64, u_2i+1, 0x64] with u = q + 128: the binary16 pair
      // (1024 + u_2i, 1024 + u_2i+1); adding -1152 to each gives (q_2i, q_2i+1)
      const uint32_t magic = prmt(w[p / 4] ^ 0x80808080u, 0x64646464u, p % 4 == 0 ? 0x4140u : 0x4342u);
      o[i] = hadd2(magic, 0xE480E480u);
    });
    tmem_st16(ta + 16u * (4 * G + t), o);
  });
}

struct TcCtx {
  ConsumerCtx cc;        // ring, parked sums, epilogue scratch, barriers, identity, unit range
  uint32_t tmem;         // tensor-memory base address
  uint32_t a_full;       // a_full[2]: every converter warp wrote unit i's A and B (count kTcWarps)
  uint32_t d_full;       // d_full[2]: unit i's MMAs completed (one tcgen05.commit)
  uint8_t *bop;          // B[2]
  float *xinv;           // [3][8][4]
};

// The converter warps' walk over the CTA's units (G: block group of the warp).
template <int N, Epi E, int G>
__device__ __forceinline__ void tc_consumer_loop(const GemvArgs &a, const TcCtx &t) {
  using S = Stage<Fmt::Q8, N>;
  constexpr int kOut = N;
  const ConsumerCtx &c = t.cc;
  const uint64_t limit = wait_limit(a);
  const uint32_t q = c.warp & 3u;
  const uint32_t row = 32u * q + c.lane;           // this thread's row of the unit
  const uint32_t tl = t.tmem + ((32u * q) << 16);  // this warp's tensor-memory lanes
  const int64_t nu = c.u1 - c.u0;
  bool scales_ready = (E == Epi::Plain) || c.warp >= static_cast<uint32_t>(kOut);
  auto wait_scales = [&]() {
    if (scales_ready) return;
    scales_ready = true;
    derive_input_scale<kOut>(a, c, limit);
  };
  auto fail = [&]() {
    if (c.flag[0] == 0) atomicOr(&g_device_error, PTI_DEVERR_FULL_TIMEOUT);
    c.flag[0] = 1;
  };
  float acc[N];
#pragma unroll
  for (int n = 0; n < N; ++n) acc[n] = 0.0f;
  float d_cur[4] = {0.0f, 0.0f, 0.0f, 0.0f}, d_prev[4] = {0.0f, 0.0f, 0.0f, 0.0f};
  uint32_t st = 0, ph = 0;  // ring slot and phase parity of the unit being converted
  // row tile and super-block of the unit being summed (one behind)
  int32_t rb = static_cast<int32_t>(c.u0 / a.n_sb);
  int32_t sb = static_cast<int32_t>(c.u0 - static_cast<int64_t>(rb) * a.n_sb);
  const int32_t rb_first = rb;
  const int32_t rb_last = static_cast<int32_t>((c.u1 - 1) / a.n_sb);

  for (int64_t i = 0; i <= nu; ++i) {
    if (i < nu) {
      // ---- convert unit i into A[i % 2], B[i % 2]
      const uint32_t s = static_cast<uint32_t>(i & 1);
      const uint32_t full = c.bars + 8 * st;
      bool ok = mbar_test_wait(full, ph);
      if (!ok) {
        ok = c.flag[0] == 0 && mbar_wait_bounded(full, ph, c.flags, limit);
        if (!ok) fail();
      }
      ok = __all_sync(0xFFFFFFFFu, ok);  // the tensor-memory stores are warp-wide
      if (ok) {
        const uint8_t *tile = c.base_ptr + st * S::kBytes;
        tc_split_x<N>(reinterpret_cast<const float *>(tile + kStageBytes), t.bop + s * kTcBBytes,
                      t.xinv + (i % 3) * 32, c.warp, c.lane);
        tc_convert<G>(tile + row * kSBBytes, tl + kTcAOff + s * 128u, d_cur);
      }
      __syncwarp();
      if (c.lane == 0) mbar_arrive(c.bars + 8 * (c.stages + st));  // the ring slot is free
      tmem_wait_st();
      fence_proxy_async_smem();  // B is read by the tensor core
      tc_fence_before();
      __syncwarp();
      if (c.lane == 0) mbar_arrive(t.a_full + 8 * s);
      if (++st == static_cast<uint32_t>(c.stages)) {
        st = 0;
        ph ^= 1u;
      }
    }
    // every warp's 2^-k of unit i - 1 (written before it reached this point
    // in the previous iteration) are visible after the barrier
    named_barrier(kBarConsumers, kTcThreads);
    if (i >= 1) {
      // ---- sum unit j = i - 1 from D[j % 2]
      const int64_t j = i - 1;
      const uint32_t s = static_cast<uint32_t>(j & 1);
      const uint32_t dbar = t.d_full + 8 * s, par = static_cast<uint32_t>((j >> 1) & 1);
      bool ok = mbar_test_wait(dbar, par);
      if (!ok) {
        ok = c.flag[0] == 0 && mbar_wait_bounded(dbar, par, c.flags, limit);
        if (!ok) fail();
      }
      ok = __all_sync(0xFFFFFFFFu, ok);  // the tensor-memory loads are warp-wide
      if (ok) {
        tc_fence_after();
        uint32_t v0[32], v1[32];
        tmem_ld32(tl + kTcDOff + s * 128u + 64u * G, v0);
        tmem_ld32(tl + kTcDOff + s * 128u + 64u * G + 32u, v1);
        const float *xi = t.xinv + (j % 3) * 32 + 16 * G;
        float p[N];
        static_for<0, 4>([&](auto b_) {
          constexpr int b = decltype(b_)::value;
          const uint32_t *v = (b < 2) ? v0 + 16 * b : v1 + 16 * (b - 2);
          const float4 xv = *reinterpret_cast<const float4 *>(xi + 4 * b);
          const float xs[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
          for (int n = 0; n < N; ++n) {
            const float val = __uint_as_float(v[3 * n]) + (__uint_as_float(v[3 * n + 1]) + __uint_as_float(v[3 * n + 2]));
            const float wv = val * d_prev[b];
            if constexpr (b == 0) p[n] = wv * xs[n];
            else p[n] = fmaf(wv, xs[n], p[n]);
          }
        });
#pragma unroll
        for (int n = 0; n < N; ++n) acc[n] += p[n];
      }
      // ---- end of a row tile: park the row's sums (slot 0 = first tile of the
      //      CTA, slot 1 = a later one) and finish the tiles wholly inside the range
      if (++sb == a.n_sb || j == nu - 1) {
        const int sl = (rb == rb_first) ? 0 : 1;
#pragma unroll
        for (int n = 0; n < N; ++n) {
          c.red[((sl * 2 + G) * kOut + n) * kRowsPerTile + row] = acc[n];
          acc[n] = 0.0f;
        }
        if (rb != rb_first && rb != rb_last) {
          wait_scales();
          named_barrier(kBarConsumers, kTcThreads);
          finish_tiles<Fmt::Q8, N, E, TcTotals<N>>(a, c.red, 1, rb, 1, 0, 0, c.tid, c.epi);
          named_barrier(kBarConsumers, kTcThreads);
        }
        sb = 0;
        ++rb;
      }
    }
#pragma unroll
    for (int b = 0; b < 4; ++b) d_prev[b] = d_cur[b];
  }
  wait_scales();
  named_barrier(kBarConsumers, kTcThreads);
  finish_tiles<Fmt::Q8, N, E, TcTotals<N>>(a, c.red, rb_last != rb_first ? 2 : 1, rb_first, 0, rb_last, 1, c.tid,
                                            c.epi);
}

// Lane 0 of the MMA warp: for each unit, once every converter warp has
// written its A and B, issue the 16 MMAs into D[i % 2] and commit them to
// d_full[i % 2].  Before returning it waits for its last MMAs, so the tensor
// memory can be released.
__device__ __forceinline__ void tc_mma_loop(const GemvArgs &a, int64_t nu, uint32_t tmem, uint32_t b_ops,
                                            uint32_t a_full, uint32_t d_full, uint32_t flags,
                                            volatile uint32_t *flag) {
  const uint64_t limit = wait_limit(a);
  int64_t issued = 0;
  for (int64_t i = 0; i < nu; ++i) {
    const uint32_t s = static_cast<uint32_t>(i & 1), par = static_cast<uint32_t>((i >> 1) & 1);
    const uint32_t bar = a_full + 8 * s;
    if (!mbar_test_wait(bar, par) && (flag[0] != 0 || !mbar_wait_bounded(bar, par, flags, limit))) {
      if (flag[0] == 0) atomicOr(&g_device_error, PTI_DEVERR_FULL_TIMEOUT);
      flag[0] = 1;
      break;
    }
    tc_fence_after();
    const uint32_t a_t = tmem + kTcAOff + s * 128u, d_t = tmem + kTcDOff + s * 128u;
    const uint32_t b_s = b_ops + s * kTcBBytes;
#pragma unroll
    for (uint32_t b = 0; b < 8; ++b) {
      mma_f16_ts(d_t + 16u * b, a_t + 16u * b, tc_smem_desc(b_s + (4u * b) * kTcLbo), kTcIdesc, 0u);
      mma_f16_ts(d_t + 16u * b, a_t + 16u * b + 8u, tc_smem_desc(b_s + (4u * b + 2u) * kTcLbo), kTcIdesc, 1u);
    }
    mma_commit(d_full + 8 * s);
    issued = i + 1;
  }
  if (issued > 0) {
    const int64_t j = issued - 1;
    if (!mbar_wait_bounded(d_full + 8 * static_cast<uint32_t>(j & 1), static_cast<uint32_t>((j >> 1) & 1), 0, limit))
      atomicOr(&g_device_error, PTI_DEVERR_DRAIN_TIMEOUT);
  }
}

// Shared memory after the ring: B[2] | xinv | parked sums | full[stages],
// empty[stages], a_full[2], d_full[2] | abort flag, tensor-memory base | the
// staged-sums barrier | fused-epilogue scratch | staged input sums.
template <int N, Epi E>
__global__ void __launch_bounds__(kTcThreads + 64, 1)
    gemv_tc_kernel(const __grid_constant__ CUtensorMap tmap, const __grid_constant__ CUtensorMap tmap2,
                   const __grid_constant__ GemvArgs a) {
  using S = Stage<Fmt::Q8, N>;
  using L = TcLayout<N>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t *const base_ptr = smem_raw + (base - raw);
  const int stages = a.stages;
  const uint32_t b_ops = base + stages * S::kBytes;
  uint8_t *const bop = base_ptr + (b_ops - base);
  float *const xinv = reinterpret_cast<float *>(bop + 2 * kTcBBytes);
  float *const red = xinv + L::kXinvBytes / 4;
  const uint32_t bars = b_ops + 2 * kTcBBytes + L::kXinvBytes + L::kRedBytes;  // full, empty
  const uint32_t a_full = bars + 16 * stages, d_full = a_full + 16;
  const uint32_t flags = d_full + 16;  // [0] abort, [1] tensor-memory base
  const uint32_t sq_bar = flags + 8;
  volatile uint32_t *const flag = reinterpret_cast<volatile uint32_t *>(base_ptr + (flags - base));
  float *const epi = reinterpret_cast<float *>(base_ptr + (flags - base) + 16);
  const uint32_t sq_stage = flags + 16 + kEpiBytes;

  const uint32_t tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t u0 = static_cast<int64_t>(blockIdx.x) * a.units / a.grid;
  const int64_t u1 = static_cast<int64_t>(blockIdx.x + 1) * a.units / a.grid;

  if (warp == kTcWarps + 1) {
    tmem_alloc(flags + 4, kTcCols);
    tmem_relinquish();
  }
  if (tid == 0) {
    for (int i = 0; i < stages; ++i) {
      mbar_init(bars + 8 * i, 1);
      mbar_init(bars + 8 * (stages + i), kTcWarps);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(a_full + 8 * s, kTcWarps);
      mbar_init(d_full + 8 * s, 1);
    }
    mbar_init(sq_bar, 1);
    flag[0] = 0;
    mbar_init_fence();
  }
  // B rows past the pieces stay zero
  for (uint32_t o = tid * 16u; o < 2u * kTcBBytes; o += blockDim.x * 16u)
    *reinterpret_cast<uint4 *>(bop + o) = make_uint4(0u, 0u, 0u, 0u);
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = flag[1];
  if (tid == 0) pdl_launch_dependents();

  if (warp == kTcWarps) {
    // ---------------- producer: one lane issues every copy --------------------
    if (lane == 0) {
      Producer<Fmt::Q8, N, E> prod{&tmap, &tmap2, &a, base, bars, flags, flag, stages, u0, u1 - u0, 0,
                                   l2_policy_evict_first(), sq_bar, sq_stage, kMaxStages, 0, 0, 0};
      prod.start();
      uint32_t st = 0, ph = 0;
      for (int64_t i = 0; i + stages < prod.nu && flag[0] == 0; ++i) {
        prod.refill(i, st, ph);
        if (++st == static_cast<uint32_t>(stages)) {
          st = 0;
          ph ^= 1u;
        }
      }
      prod.drain();
    }
    return;
  }
  if (warp == kTcWarps + 1) {
    // ---------------- MMA issue; owner of the tensor memory ------------------
    if (lane == 0) tc_mma_loop(a, u1 - u0, tmem, b_ops, a_full, d_full, flags, flag);
    __syncwarp();
    named_barrier(kBarTcExit, kTcThreads + 32);
    tc_fence_after();
    tmem_dealloc(tmem, kTcCols);
    return;
  }

  // ---------------- converter warps ------------------------------------------
  const TcCtx t{ConsumerCtx{base_ptr, red, epi, flag, bars, flags, sq_bar, sq_stage, stages, tid, warp, lane, u0, u1},
                tmem, a_full, d_full, bop, xinv};
  if (warp < 4) tc_consumer_loop<N, E, 0>(a, t);
  else tc_consumer_loop<N, E, 1>(a, t);
  tc_fence_before();
  named_barrier(kBarTcExit, kTcThreads + 32);
}
