// NF4 constants of the device code: the 16 levels and the 15 decision
// thresholds, as float32 bit patterns.
//
// Levels: the NormalFloat-4 construction of the QLoRA paper (normal quantiles
// at 9 evenly spaced probabilities from 1 - (1/30 + 1/32)/2 to 1/2 for the 8
// positive levels, 8 such probabilities for the 7 negative ones, plus 0;
// normalised by the largest and rounded to float32).
// Threshold j: the smallest float32 strictly greater than the exact midpoint
// (T[j] + T[j+1]) / 2, so that  code = #{ j : x >= thr[j] }  is the nearest
// level to x with ties going to the lower level.
#pragma once
#include <stdint.h>

#define SL_NF4_LEVEL_BITS                                                                                  \
  0xbf800000u, 0xbf3239b1u, 0xbf066b2eu, 0xbeca329eu, 0xbe91a24bu, 0xbe3d353du, 0xbdba7869u, 0x00000000u, \
      0x3da2fb01u, 0x3e24cadfu, 0x3e7c04dau, 0x3ead0336u, 0x3ee1a4b5u, 0x3f1007a9u, 0x3f3913b0u, 0x3f800000u

#define SL_NF4_THRESH_BITS                                                                                 \
  0xbf591cd8u, 0xbf1c526fu, 0xbeeb847cu, 0xbeadea74u, 0xbe703ce9u, 0xbe0d38b8u, 0xbd3a7868u, 0x3d22fb02u, \
      0x3df64860u, 0x3e5067ddu, 0x3e9582d2u, 0x3ec753f6u, 0x3f006d02u, 0x3f248dadu, 0x3f5c89d9u

namespace sl {

static constexpr uint32_t kNF4LevelBits[16] = {SL_NF4_LEVEL_BITS};
static constexpr uint32_t kNF4ThreshBits[15] = {SL_NF4_THRESH_BITS};

// Device copies (one per translation unit that uses them).
static __device__ __constant__ uint32_t d_nf4_level_bits[16] = {SL_NF4_LEVEL_BITS};
static __device__ __constant__ uint32_t d_nf4_thresh_bits[15] = {SL_NF4_THRESH_BITS};

}  // namespace sl
