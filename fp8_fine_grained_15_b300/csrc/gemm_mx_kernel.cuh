// MX (microscaling) FP8 GEMM: C = A * B^T over E4M3 operands with one
// power-of-two (UE8M0) scale per 32-deep K group of every row of A and of B,
// applied by the tensor cores themselves -- the direction the pages point to
// after 1x128 / 128x128 scaling ("Should Fixing Deepseek Take 60 Steps?",
// Figure 7 (a) passage; page at why-be.why-be.co.kr, accumulation-precision
// passage: group scaling moves into the MMA on the next GPU generation).
//
// With the scales inside tcgen05.mma (kind::mxf8f6f4, block_scale,
// scale_vec::1X) there is no promotion on CUDA cores: the MMAs of a whole
// tile accumulate in one TMEM buffer across all of K and the CUDA cores only
// run the epilogue.
//
// B300 design (one CTA per SM, persistent over 128 x 256 output tiles, m
// tiles fastest):
//   warp 0      TMA producer: per 128-deep K block, the A tile (128 x 128 B),
//               the B tile (256 x 128 B), 128-byte swizzle, and the exponent
//               words of its 128 rows of A and 256 rows of B (one 32-bit word
//               = the four group exponents of a row in this K block), into a
//               4-stage ring.
//   warp 1      MMA issuer: 4 x block-scaled MMA (M=128, N=256, K=32) per K
//               block into the accumulator (TMEM columns 0..255); MMA kk reads
//               byte kk of every scale cell.
//   warps 4..7  scale writers: copy the stage's exponent words from shared
//               memory into the stage's TMEM scale slot with tcgen05.st, each
//               warp into its own lane quadrant (the layout below), then
//               signal the MMA issuer.
//   warps 8..15 epilogue: tcgen05.ld of the finished tile (32 rows x 128
//               columns per warp), release the accumulator, BF16 / FP32
//               through shared memory and TMA stores.
// TMEM scale layout of one slot (16 columns at 256 + 16 * stage): the scale
// word of A row r (0..127 within the tile) sits in lane r % 32 of every lane
// quadrant, column r / 32 (4 columns); that of B row n (0..255) in lane n % 32
// of every quadrant, column 4 + n / 32 (8 columns).
#pragma once
#include <cuda_bf16.h>

#include <cstdint>

#include "gemm_kernel.cuh"
#include "ptx.cuh"

namespace fp8bs {

constexpr int kMxStages = 4;
constexpr int kMxThreads = 512;        // 4 warpgroups
constexpr int kMxEpiWarps = 8;
constexpr uint32_t kMxTmemCols = 512;  // accumulator 0..255, scale slots from 256
constexpr uint32_t kMxSfCol0 = 256;
constexpr uint32_t kMxSfPitch = 16;    // columns per scale slot: 4 (A) + 8 (B), padded
constexpr uint32_t kMxSfBytes = (kBM + kBN) * 4;
// Register split: launch budget 128 x 512; producers keep 40, scale writers
// 64, the two epilogue warpgroups 200 (128*40 + 128*64 + 256*200 = 64512).
constexpr uint32_t kMxProducerRegs = 40;
constexpr uint32_t kMxSfRegs = 64;
constexpr uint32_t kMxEpilogueRegs = 200;
static_assert(128 * kMxProducerRegs + 128 * kMxSfRegs + 256 * kMxEpilogueRegs <= 128 * kMxThreads,
              "register split exceeds the launch budget");
static_assert(kMxSfCol0 + kMxStages * kMxSfPitch <= kMxTmemCols, "scale slots exceed TMEM");

struct MxParams {
  int32_t M, N, KB, num_m_tiles, num_n_tiles;
};

struct MxSmem {
  alignas(1024) unsigned char epi_stage[kMxEpiWarps][kEpiStageBytes];
  alignas(128) uint32_t sfa[kMxStages][kBM];   // exponent words of the stage's A rows
  alignas(128) uint32_t sfb[kMxStages][kBN];   // ... and of its B rows
  uint64_t full[kMxStages];
  uint64_t empty[kMxStages];
  uint64_t sf_full[kMxStages];
  uint64_t acc_full;
  uint64_t acc_empty;
  uint64_t drain;
  uint32_t tmem_base;
  int32_t abort_flag;
};

constexpr size_t kMxSmemBytes =
    1024 /* alignment slack */ + static_cast<size_t>(kMxStages) * kStageBytes + sizeof(MxSmem);

template <bool kOutBf16>
__global__ void __launch_bounds__(kMxThreads, 1)
    fp8bs_mx_gemm_kernel(const __grid_constant__ MxParams p,
                         const __grid_constant__ CUtensorMap tmap_a,
                         const __grid_constant__ CUtensorMap tmap_b,
                         const __grid_constant__ CUtensorMap tmap_sfa,
                         const __grid_constant__ CUtensorMap tmap_sfb,
                         const __grid_constant__ CUtensorMap tmap_c) {
  extern __shared__ __align__(1024) unsigned char mx_smem_raw[];
  const uint32_t raw_addr = smem_u32(mx_smem_raw);
  unsigned char* ring = mx_smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  MxSmem& sm = *reinterpret_cast<MxSmem*>(ring + static_cast<size_t>(kMxStages) * kStageBytes);
  const uint32_t ring_addr = smem_u32(ring);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  volatile int* abort_flag = &sm.abort_flag;
  const int num_tiles = p.num_m_tiles * p.num_n_tiles;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kMxStages; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], 1);
      mbar_init(&sm.sf_full[s], 4);
    }
    mbar_init(&sm.acc_full, 1);
    mbar_init(&sm.acc_empty, kMxEpiWarps);
    mbar_init(&sm.drain, 1);
    sm.abort_flag = 0;
    fence_mbarrier_init();
    tma_prefetch_desc(&tmap_a);
    tma_prefetch_desc(&tmap_b);
    tma_prefetch_desc(&tmap_sfa);
    tma_prefetch_desc(&tmap_sfb);
    tma_prefetch_desc(&tmap_c);
  }
  if (warp == 1) tmem_alloc(&sm.tmem_base, kMxTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = sm.tmem_base;

  if (warp < 4) {
    regs_dealloc<kMxProducerRegs>();
    if (warp == 0 && lane == 0) {
      // ---------------------------------------------------------------- TMA
      const uint64_t policy = l2_policy_evict_last();
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued_mask = 0, parity_mask = 0;
      for (int t = blockIdx.x; t < num_tiles; t += gridDim.x) {
        const int m0 = (t % p.num_m_tiles) * kBM;
        const int n0 = (t / p.num_m_tiles) * kBN;
        for (int kb = 0; kb < p.KB; ++kb) {
          if (!bounded_wait(&sm.empty[stage], phase ^ 1u, abort_flag)) goto producer_done;
          mbar_arrive_expect_tx(&sm.full[stage], kStageBytes + kMxSfBytes);
          const uint32_t sa_addr = ring_addr + stage * kStageBytes;
          tma_load_2d(sa_addr, &tmap_a, kb * kBK, m0, &sm.full[stage], policy);
          tma_load_2d(sa_addr + kStageABytes, &tmap_b, kb * kBK, n0, &sm.full[stage], policy);
          tma_load_2d(smem_u32(&sm.sfa[stage][0]), &tmap_sfa, m0, kb, &sm.full[stage], policy);
          tma_load_2d(smem_u32(&sm.sfb[stage][0]), &tmap_sfb, n0, kb, &sm.full[stage], policy);
          issued_mask |= 1u << stage;
          parity_mask = (parity_mask & ~(1u << stage)) | (phase << stage);
          if (++stage == kMxStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
    producer_done:
      for (int s = 0; s < kMxStages; ++s)
        if (issued_mask & (1u << s))
          bounded_wait_noabort(&sm.full[s], (parity_mask >> s) & 1u, kSpinLimitNs);
    } else if (warp == 1 && lane == 0) {
      // ---------------------------------------------------------------- MMA
      int stage = 0;
      uint32_t phase = 0, aphase = 0;
      bool issued = false;
      for (int t = blockIdx.x; t < num_tiles; t += gridDim.x) {
        // the epilogue must have read the previous tile out of the accumulator
        if (!bounded_wait(&sm.acc_empty, aphase ^ 1u, abort_flag)) goto mma_done;
        tc_fence_after();
        for (int kb = 0; kb < p.KB; ++kb) {
          if (!bounded_wait(&sm.full[stage], phase, abort_flag)) goto mma_done;
          if (!bounded_wait(&sm.sf_full[stage], phase, abort_flag)) goto mma_done;
          tc_fence_after();
          const uint32_t a_addr = ring_addr + stage * kStageBytes;
          const uint64_t adesc = smem_desc_k_sw128(a_addr);
          const uint64_t bdesc = smem_desc_k_sw128(a_addr + kStageABytes);
          const uint32_t sfa_t = tmem_base + kMxSfCol0 + static_cast<uint32_t>(stage) * kMxSfPitch;
#pragma unroll
          for (int kk = 0; kk < kBK / 32; ++kk)
            mma_mxf8f6f4(tmem_base, adesc + 2u * kk, bdesc + 2u * kk,
                         idesc_mx_e4m3(kBM, kBN, static_cast<uint32_t>(kk)), sfa_t, sfa_t + 4u,
                         (kb > 0 || kk > 0) ? 1u : 0u);
          mma_commit(&sm.empty[stage]);
          issued = true;
          if (++stage == kMxStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        mma_commit(&sm.acc_full);
        aphase ^= 1u;
      }
    mma_done:
      if (issued) {
        mma_commit(&sm.drain);
        bounded_wait_noabort(&sm.drain, 0, kSpinLimitNs);
      }
    }
  } else if (warp < 8) {
    regs_dealloc<kMxSfRegs>();
    // ------------------------------------------------------- scale writers
    // A full stage also means the MMAs that last read this slot are done:
    // the producer refilled the stage only after their commit.
    const uint32_t quad = static_cast<uint32_t>(warp & 3) * 32u;
    int stage = 0;
    uint32_t phase = 0;
    for (int t = blockIdx.x; t < num_tiles; t += gridDim.x) {
      for (int kb = 0; kb < p.KB; ++kb) {
        if (!bounded_wait(&sm.full[stage], phase, abort_flag)) goto writers_done;
        tc_fence_after();
        uint32_t a[4], b[8];
#pragma unroll
        for (int c = 0; c < 4; ++c) a[c] = sm.sfa[stage][32 * c + lane];
#pragma unroll
        for (int c = 0; c < 8; ++c) b[c] = sm.sfb[stage][32 * c + lane];
        const uint32_t taddr =
            tmem_base + (quad << 16) + kMxSfCol0 + static_cast<uint32_t>(stage) * kMxSfPitch;
        tmem_st4(taddr, a);
        tmem_st8(taddr + 4u, b);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.sf_full[stage]);
        if (++stage == kMxStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
  writers_done:;
  } else {
    regs_alloc<kMxEpilogueRegs>();
    // ------------------------------------------------------------ epilogue
    const int g = warp & 3;          // TMEM lane quadrant (rows 32g .. 32g+31)
    const int h = (warp - 8) >> 2;   // column half (0: 0..127, 1: 128..255)
    uint32_t aphase = 0;
    for (int t = blockIdx.x; t < num_tiles; t += gridDim.x) {
      const int m0 = (t % p.num_m_tiles) * kBM;
      const int n0 = (t / p.num_m_tiles) * kBN;
      if (!bounded_wait(&sm.acc_full, aphase, abort_flag)) goto epilogue_done;
      tc_fence_after();
      float2 acc[64];
      const uint32_t taddr =
          tmem_base + (static_cast<uint32_t>(g * 32) << 16) + static_cast<uint32_t>(h * 128);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t r[32];
        tmem_ld32(taddr + c * 32, r);
        tmem_wait_ld(r);
#pragma unroll
        for (int i = 0; i < 16; ++i)
          acc[c * 16 + i] = make_float2(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1]));
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.acc_empty);
      aphase ^= 1u;
      const int col0 = n0 + h * 128;
      if (col0 < p.N)
        store_rows_tma<kOutBf16>(acc, smem_u32(&sm.epi_stage[warp - 8][0]), lane, &tmap_c, col0,
                                 m0 + g * 32);
    }
  epilogue_done:
    if (lane == 0) bulk_wait_all();
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc(tmem_base, kMxTmemCols);
  }
}

}  // namespace fp8bs
