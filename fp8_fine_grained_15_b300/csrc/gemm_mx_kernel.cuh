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
// B300 design: clusters of two CTAs (tcgen05 cta_group::2), persistent over
// 256 x 256 output tiles, m tiles fastest (the kernel is described below).
// TMEM scale layout of one slot (16 columns at 256 + 16 * stage): the scale
// word of A row r (0..127 within the CTA's half of the tile) sits in lane
// r % 32 of every lane quadrant, column r / 32 (4 columns); that of B row n
// (0..255 within the tile) in lane n % 32 of every quadrant, column 4 + n / 32
// (8 columns).  Each CTA holds the words of its own A rows and of all 256 B
// rows: planted single-group GEMMs (every row and column with its own
// exponent per group) come out exact on both CTAs of a pair tile.
#pragma once
#include <cuda_bf16.h>

#include <cstdint>

#include "gemm_kernel.cuh"
#include "gemm_pair_kernel.cuh"
#include "ptx.cuh"

namespace fp8bs {

constexpr int kMxThreads = 512;        // 4 warpgroups
constexpr int kMxEpiWarps = 8;
constexpr uint32_t kMxTmemCols = 512;  // accumulator 0..255, scale slots from 256
constexpr uint32_t kMxSfCol0 = 256;
constexpr uint32_t kMxSfPitch = 16;    // columns per scale slot: 4 (A) + 8 (B), padded
// Register split: launch budget 128 x 512; producers keep 40, scale writers
// 64, the two epilogue warpgroups 200 (128*40 + 128*64 + 256*200 = 64512).
constexpr uint32_t kMxProducerRegs = 40;
constexpr uint32_t kMxSfRegs = 64;
constexpr uint32_t kMxEpilogueRegs = 200;
static_assert(128 * kMxProducerRegs + 128 * kMxSfRegs + 256 * kMxEpilogueRegs <= 128 * kMxThreads,
              "register split exceeds the launch budget");

struct MxParams {
  int32_t M, N, KB, num_m_tiles, num_n_tiles;
};

// ------------------------------------------------------------ CTA pairs
// A 256 x 256 output tile per cluster of two CTAs, each CTA staging its own
// 128 rows of A and one half (128 rows) of the B tile, so every SM pulls 32 KB
// of operands per K block (one CTA per 128 x 256 tile pulled 48 KB with four
// stages: 0.358 -> 0.348 ms on the layer's Fprop shape, same-box A/B) and six
// stages fit in shared memory.  The even CTA issues
// the block-scaled pair MMAs.  Each CTA's tensor core reads the scale cells
// from its own TMEM: the A words of its own 128 rows and the B words of all
// 256 B rows of the tile (the single-CTA slot layout), so each CTA loads the
// tile's 256 B words.
//   warp 0      TMA producer (both CTAs): A rows and B half with cta_group::2
//               copies that complete on the even CTA's `full` barrier; the
//               exponent words with plain copies on the CTA's own `sf_data`
//               barrier.
//   warp 1      even CTA: 4 x pair MMA (M=256, N=256, K=32) per K block, one
//               commit to `done` in both CTAs; after a tile's last K block a
//               commit to `acc_full` in both CTAs.
//   warps 4..7  scale writers (both CTAs): words into the CTA's TMEM slot,
//               then an arrive on the even CTA's `sf_full` (8 arrivals).
//   warps 8..15 epilogue (both CTAs): read the CTA's 128 rows out of the
//               accumulator, arrive on the even CTA's `acc_empty` (16
//               arrivals), then the TMA-store epilogue.
constexpr int kMxPairStages = 6;
constexpr int kMxPairStageA = kBM * kBK;           // this CTA's 128 rows of A, one K block
constexpr int kMxPairStageB = (kBN / 2) * kBK;     // this CTA's half of the B tile
constexpr int kMxPairStageBytes = kMxPairStageA + kMxPairStageB;
constexpr uint32_t kMxPairSfBytes = (kBM + kBN) * 4;   // A words of 128 rows, B words of 256
static_assert(kMxSfCol0 + kMxPairStages * kMxSfPitch <= kMxTmemCols, "scale slots exceed TMEM");

struct MxPairSmem {
  alignas(1024) unsigned char epi_stage[kMxEpiWarps][kEpiStageBytes];
  alignas(128) uint32_t sfa[kMxPairStages][kBM];   // exponent words of this CTA's A rows
  alignas(128) uint32_t sfb[kMxPairStages][kBN];   // ... and of all the tile's B rows
  uint64_t full[kMxPairStages];      // even CTA: both CTAs' operand copies landed
  uint64_t done[kMxPairStages];      // both CTAs: the K block's MMAs are complete
  uint64_t sf_data[kMxPairStages];   // this CTA's exponent words landed
  uint64_t sf_full[kMxPairStages];   // even CTA: both CTAs' scale slots are written
  uint64_t acc_full;                 // both CTAs: the tile's accumulator is final
  uint64_t acc_empty;                // even CTA: both CTAs' epilogues have read it
  uint64_t drain;
  uint32_t tmem_base;
  int32_t abort_flag;
};

constexpr size_t kMxPairSmemBytes = 1024 /* alignment slack */ +
                                    static_cast<size_t>(kMxPairStages) * kMxPairStageBytes +
                                    sizeof(MxPairSmem);

// p.num_m_tiles counts 256-row pair tiles.
template <bool kOutBf16>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kMxThreads, 1)
    fp8bs_mx_gemm_pair_kernel(const __grid_constant__ MxParams p,
                              const __grid_constant__ CUtensorMap tmap_a,
                              const __grid_constant__ CUtensorMap tmap_b,
                              const __grid_constant__ CUtensorMap tmap_sfa,
                              const __grid_constant__ CUtensorMap tmap_sfb,
                              const __grid_constant__ CUtensorMap tmap_c) {
  extern __shared__ __align__(1024) unsigned char mxp_smem_raw[];
  const uint32_t raw_addr = smem_u32(mxp_smem_raw);
  unsigned char* ring = mxp_smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  MxPairSmem& sm =
      *reinterpret_cast<MxPairSmem*>(ring + static_cast<size_t>(kMxPairStages) * kMxPairStageBytes);
  const uint32_t ring_addr = smem_u32(ring);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();   // 0: the CTA that issues the MMAs
  volatile int* abort_flag = &sm.abort_flag;
  const int num_tiles = p.num_m_tiles * p.num_n_tiles;
  const int first = static_cast<int>(blockIdx.x >> 1);
  const int stride = static_cast<int>(gridDim.x >> 1);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kMxPairStages; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.done[s], 1);
      mbar_init(&sm.sf_data[s], 1);
      mbar_init(&sm.sf_full[s], 8);
    }
    mbar_init(&sm.acc_full, 1);
    mbar_init(&sm.acc_empty, 2 * kMxEpiWarps);
    mbar_init(&sm.drain, 1);
    sm.abort_flag = 0;
    fence_mbarrier_init();
    tma_prefetch_desc(&tmap_a);
    tma_prefetch_desc(&tmap_b);
    tma_prefetch_desc(&tmap_sfa);
    tma_prefetch_desc(&tmap_sfb);
    tma_prefetch_desc(&tmap_c);
  }
  if (warp == 1) tmem_alloc_pair(&sm.tmem_base, kMxTmemCols);
  tc_fence_before();
  __syncwarp();
  cluster_sync();   // barriers of both CTAs initialised, TMEM allocated in both
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
      bool aborted = false;
      for (int t = first; t < num_tiles && !aborted; t += stride) {
        const int mt = t % p.num_m_tiles, nt = t / p.num_m_tiles;
        const int a_row = mt * kPairTileM + static_cast<int>(rank) * kBM;
        const int b_row = nt * kBN + static_cast<int>(rank) * (kBN / 2);
        for (int kb = 0; kb < p.KB; ++kb) {
          if (!bounded_wait(&sm.done[stage], phase ^ 1u, abort_flag)) {
            aborted = true;
            break;
          }
          if (rank == 0) mbar_arrive_expect_tx(&sm.full[stage], 2 * kMxPairStageBytes);
          const uint32_t full_bar = mapa_shared(smem_u32(&sm.full[stage]), 0);
          const uint32_t dst = ring_addr + stage * kMxPairStageBytes;
          tma_load_2d_pair(dst, &tmap_a, kb * kBK, a_row, full_bar, policy);
          tma_load_2d_pair(dst + kMxPairStageA, &tmap_b, kb * kBK, b_row, full_bar, policy);
          mbar_arrive_expect_tx(&sm.sf_data[stage], kMxPairSfBytes);
          tma_load_2d(smem_u32(&sm.sfa[stage][0]), &tmap_sfa, a_row, kb, &sm.sf_data[stage], policy);
          tma_load_2d(smem_u32(&sm.sfb[stage][0]), &tmap_sfb, nt * kBN, kb, &sm.sf_data[stage],
                      policy);
          issued_mask |= 1u << stage;
          parity_mask = (parity_mask & ~(1u << stage)) | (phase << stage);
          if (++stage == kMxPairStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // Every copy issued must land before either CTA may exit: the even CTA
      // sees both CTAs' operand bytes on `full`; each CTA sees its own words
      // on `sf_data` (the odd CTA's operand copies land with them or, after an
      // abort, within the sleep).
      for (int s = 0; s < kMxPairStages; ++s)
        if (issued_mask & (1u << s)) {
          if (rank == 0) bounded_wait_noabort(&sm.full[s], (parity_mask >> s) & 1u, kSpinLimitNs);
          bounded_wait_noabort(&sm.sf_data[s], (parity_mask >> s) & 1u, kSpinLimitNs);
        }
      if (rank != 0 && aborted) __nanosleep(100000);
    } else if (warp == 1 && lane == 0 && rank == 0) {
      // ---------------------------------------------------------------- MMA
      int stage = 0;
      uint32_t phase = 0, aphase = 0;
      bool issued = false;
      for (int t = first; t < num_tiles; t += stride) {
        // both CTAs' epilogues must have read the previous tile
        if (!bounded_wait(&sm.acc_empty, aphase ^ 1u, abort_flag)) goto mma_done;
        tc_fence_after();
        for (int kb = 0; kb < p.KB; ++kb) {
          if (!bounded_wait(&sm.full[stage], phase, abort_flag)) goto mma_done;
          if (!bounded_wait(&sm.sf_full[stage], phase, abort_flag)) goto mma_done;
          tc_fence_after();
          const uint32_t a_addr = ring_addr + stage * kMxPairStageBytes;
          const uint64_t adesc = smem_desc_k_sw128(a_addr);
          const uint64_t bdesc = smem_desc_k_sw128(a_addr + kMxPairStageA);
          const uint32_t sfa_t = tmem_base + kMxSfCol0 + static_cast<uint32_t>(stage) * kMxSfPitch;
#pragma unroll
          for (int kk = 0; kk < kBK / 32; ++kk)
            mma_mxf8f6f4_pair(tmem_base, adesc + 2u * kk, bdesc + 2u * kk,
                              idesc_mx_e4m3(kPairTileM, kBN, static_cast<uint32_t>(kk)), sfa_t,
                              sfa_t + 4u, (kb > 0 || kk > 0) ? 1u : 0u);
          mma_commit_pair(&sm.done[stage], 0x3);
          issued = true;
          if (++stage == kMxPairStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        mma_commit_pair(&sm.acc_full, 0x3);
        aphase ^= 1u;
      }
    mma_done:
      if (issued) {  // all MMAs must finish before TMEM is released in either CTA
        mma_commit_pair(&sm.drain, 0x1);
        bounded_wait_noabort(&sm.drain, 0, kSpinLimitNs);
      }
    }
  } else if (warp < 8) {
    regs_dealloc<kMxSfRegs>();
    // ------------------------------------------------------- scale writers
    // The words of a stage land only after the MMAs that last read this
    // slot completed (the producer refilled the stage after their commit).
    const uint32_t quad = static_cast<uint32_t>(warp & 3) * 32u;
    const uint32_t sf_full0 = mapa_shared(smem_u32(&sm.sf_full[0]), 0);
    int stage = 0;
    uint32_t phase = 0;
    for (int t = first; t < num_tiles; t += stride) {
      for (int kb = 0; kb < p.KB; ++kb) {
        if (!bounded_wait(&sm.sf_data[stage], phase, abort_flag)) goto writers_done;
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
        if (lane == 0) mbar_arrive_cluster(sf_full0 + 8u * static_cast<uint32_t>(stage));
        if (++stage == kMxPairStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
  writers_done:;
  } else {
    regs_alloc<kMxEpilogueRegs>();
    // ------------------------------------------------------------ epilogue
    const int g = warp & 3;          // TMEM lane quadrant (rows 32g .. 32g+31 of this CTA)
    const int h = (warp - 8) >> 2;   // column half (0: 0..127, 1: 128..255)
    const uint32_t acc_empty0 = mapa_shared(smem_u32(&sm.acc_empty), 0);
    uint32_t aphase = 0;
    for (int t = first; t < num_tiles; t += stride) {
      const int mt = t % p.num_m_tiles, nt = t / p.num_m_tiles;
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
      if (lane == 0) mbar_arrive_cluster(acc_empty0);
      aphase ^= 1u;
      const int col0 = nt * kBN + h * 128;
      if (col0 < p.N)
        store_rows_tma<kOutBf16>(acc, smem_u32(&sm.epi_stage[warp - 8][0]), lane, &tmap_c, col0,
                                 mt * kPairTileM + static_cast<int>(rank) * kBM + g * 32);
    }
  epilogue_done:
    if (lane == 0) bulk_wait_all();
  }

  tc_fence_before();
  __syncwarp();
  cluster_sync();   // no CTA leaves while its peer may still touch its shared memory
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc_pair(tmem_base, kMxTmemCols);
  }
}

}  // namespace fp8bs
