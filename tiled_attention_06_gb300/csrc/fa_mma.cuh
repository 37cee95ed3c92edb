// The MMA blocks shared by the forward and backward kernels: a 128-row tile times a
// K/V-shaped tile, with the A operand from shared memory (issue_qk) or from TMEM
// (issue_pv). Both take 16-bit operands in 128-byte-swizzled shared memory as the TMA
// tile loads leave them.
#pragma once

#include <cstdint>

#include "fa_ptx.cuh"

namespace fa {

constexpr int kMmaM = 128;  // rows of one tcgen05 M=128 tile (= TMEM lanes)

// S = Q K^T for one 128-row tile: D/16 MMAs of K = 16, both operands K-major in
// 128-byte-swizzled shared memory (rows of 128 bytes, 8-row groups 1024 bytes apart,
// one region per 64 elements of d). The descriptors are built once; each MMA adds a
// compile-time offset to the start-address field (addresses stay below 256 KB, so the
// 14-bit field never carries), which keeps the issuing thread's dependency chain short.
// ACC: add to S instead of overwriting it.
template <int D, int BN, bool BF16, bool ACC = false>
__device__ __forceinline__ void issue_qk(uint32_t d_tmem, uint32_t q_smem, uint32_t k_smem) {
  constexpr uint32_t id = idesc_f16(BF16, kMmaM, BN, false);
  const uint64_t a0 = smem_desc_sw128(q_smem, 16, 1024);
  const uint64_t b0 = smem_desc_sw128(k_smem, 16, 1024);
  if constexpr (D == 128) {
    constexpr int QC = kMmaM * 128 / 16, KC = BN * 128 / 16;  // next 64-element region
    umma_ss8<2, 4, 6, QC, QC + 2, QC + 4, QC + 6, 2, 4, 6, KC, KC + 2, KC + 4, KC + 6, ACC>(
        d_tmem, a0, b0, id);
  } else {
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk)
      umma_ss(d_tmem, a0 + static_cast<uint64_t>(kk * 2), b0 + static_cast<uint64_t>(kk * 2), id,
              (ACC || kk > 0) ? 1u : 0u);
  }
}

// O (+)= P V: A = P from TMEM (BN/2 packed columns), B = V (BN keys x D) MN-major in
// shared memory: 16 keys per MMA = two 8-row groups (1024 bytes apart), the second
// 64-element half of d one region (BN*128 bytes) further.
template <int D, int BN, bool BF16>
__device__ __forceinline__ void issue_pv(uint32_t o_tmem, uint32_t p_tmem, uint32_t v_smem,
                                         bool accumulate) {
  constexpr uint32_t id = idesc_f16(BF16, kMmaM, D, true);
  const uint64_t b0 = smem_desc_sw128(v_smem, BN * 128, 1024);
  if constexpr (BN == 128) {
    umma_ts8<16 * 128 / 16>(o_tmem, p_tmem, b0, id, accumulate ? 1u : 0u);
  } else {
#pragma unroll
    for (int kk = 0; kk < BN / 16; ++kk)
      umma_ts(o_tmem, p_tmem + kk * 8, b0 + static_cast<uint64_t>(kk * 128), id,
              (accumulate || kk > 0) ? 1u : 0u);
  }
}

}  // namespace fa

namespace fa {

// The same two products for a 64-row query tile (tcgen05 M = 64, BLOCK_M = 64 work items).
// S = Q K^T: Q a 64-row tile (regions of 64 elements of d, 8 KB apart), K as in issue_qk.
template <int D, int BN, bool BF16>
__device__ __forceinline__ void issue_qk_m64(uint32_t d_tmem, uint32_t q_smem, uint32_t k_smem) {
  constexpr uint32_t id = idesc_f16(BF16, 64, BN, false);
  const uint64_t a0 = smem_desc_sw128(q_smem, 16, 1024);
  const uint64_t b0 = smem_desc_sw128(k_smem, 16, 1024);
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint64_t a_off = static_cast<uint64_t>((kk / 4) * (64 * 128 / 16) + (kk % 4) * 2);
    const uint64_t b_off = static_cast<uint64_t>((kk / 4) * (BN * 128 / 16) + (kk % 4) * 2);
    umma_ss(d_tmem, a0 + a_off, b0 + b_off, id, kk > 0 ? 1u : 0u);
  }
}

// O (+)= P V for a 64-row tile with P in shared memory: P [64 x BN] 16-bit, K-major,
// 128-byte swizzled (regions of 64 keys, 8 KB apart); V [BN x D] MN-major as in issue_pv.
template <int D, int BN, bool BF16>
__device__ __forceinline__ void issue_pv_m64(uint32_t o_tmem, uint32_t p_smem, uint32_t v_smem,
                                             bool accumulate) {
  constexpr uint32_t id = idesc_f16(BF16, 64, D, true);
  const uint64_t a0 = smem_desc_sw128(p_smem, 16, 1024);
  const uint64_t b0 = smem_desc_sw128(v_smem, BN * 128, 1024);
#pragma unroll
  for (int kk = 0; kk < BN / 16; ++kk) {
    const uint64_t a_off = static_cast<uint64_t>((kk / 4) * (64 * 128 / 16) + (kk % 4) * 2);
    umma_ss(o_tmem, a0 + a_off, b0 + static_cast<uint64_t>(kk * 128), id,
            (accumulate || kk > 0) ? 1u : 0u);
  }
}

}  // namespace fa
