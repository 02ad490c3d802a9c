// Constant tables of the TurboQuant codec for the CUDA kernels.
//
// Data printed on the page "mlx-bun 0.0.9 -> 0.0.11", file
// package/src/mlx/turboquant-tables.ts: SIGN_VECTORS (the +-1 rotation signs
// for head_dim 64/128/256/512) and LLOYD_MAX (value centroids and decision
// boundaries for 2/3/4/5/8 bits). Written here as exact hexadecimal float
// literals, and the signs as bitmasks: bit j of byte k is set when element
// 8k+j has sign -1.
#pragma once
#include <cstdint>

namespace tq {

__device__ const uint8_t kSignNeg64[8] = {
    0x8e, 0x54, 0x69, 0xb7, 0x02, 0x48, 0xde, 0x62,
};

__device__ const uint8_t kSignNeg128[16] = {
    0x0d, 0xdf, 0x39, 0x6a, 0x50, 0x02, 0x9c, 0x6a, 0xd5, 0x37, 0x83, 0x4a, 0xde, 0x59, 0x60, 0x14,
};

__device__ const uint8_t kSignNeg256[32] = {
    0x12, 0x30, 0xe6, 0x62, 0x11, 0x4a, 0xcd, 0x10, 0x6f, 0x14, 0x6d, 0xa9, 0xc9, 0x5e, 0x9c, 0xd3,
    0x9b, 0xf2, 0x2f, 0x3a, 0x73, 0x5d, 0x27, 0xb2, 0x6b, 0xd9, 0x30, 0x57, 0x57, 0xc3, 0x8b, 0xfe,
};

__device__ const uint8_t kSignNeg512[64] = {
    0xbd, 0x4b, 0x36, 0x70, 0x0d, 0xe3, 0xfb, 0x62, 0x63, 0xe4, 0x39, 0xd4, 0x61, 0xd2, 0xca, 0x5c,
    0x8f, 0x7c, 0x47, 0x9b, 0x43, 0x12, 0xdd, 0xe9, 0x30, 0xde, 0x2a, 0x54, 0xba, 0xca, 0xba, 0x77,
    0x84, 0x3e, 0x87, 0x11, 0x18, 0x15, 0x4c, 0x9a, 0xc5, 0xa3, 0x04, 0x32, 0x1f, 0x72, 0x81, 0x5d,
    0x52, 0x14, 0x82, 0x8a, 0xc2, 0x9b, 0xa7, 0x8e, 0xef, 0x4b, 0x0e, 0x52, 0x6d, 0x9d, 0x6b, 0x29,
};

__device__ const float kCentroids2[4] = {
    -0x1.83b4a20000000p+0f, -0x1.d538fe0000000p-2f, 0x1.cb66440000000p-2f, 0x1.831c660000000p+0f,
};

struct LloydMax2 {
  static constexpr int kBits = 2;
  // decision boundary j (ascending), j = 0 .. 2
  __host__ __device__ static constexpr float boundary(int j) {
    switch (j) {
      case 0: return -0x1.f902e20000000p-1f;
      case 1: return -0x1.3a57400000000p-8f;
      case 2: return 0x1.f5f5f80000000p-1f;
      default: return 0.0f;
    }
  }
};

__device__ const float kCentroids3[8] = {
    -0x1.1373180000000p+1f, -0x1.580a7c0000000p+0f, -0x1.8313be0000000p-1f, -0x1.f5f1be0000000p-3f,
    0x1.f5f1be0000000p-3f, 0x1.8313be0000000p-1f, 0x1.580a7c0000000p+0f, 0x1.1373180000000p+1f,
};

struct LloydMax3 {
  static constexpr int kBits = 3;
  // decision boundary j (ascending), j = 0 .. 6
  __host__ __device__ static constexpr float boundary(int j) {
    switch (j) {
      case 0: return -0x1.bf78580000000p+0f;
      case 1: return -0x1.0cca2e0000000p+0f;
      case 2: return -0x1.0048160000000p-1f;
      case 3: return 0x0.0p+0f;
      case 4: return 0x1.0048160000000p-1f;
      case 5: return 0x1.0cca2e0000000p+0f;
      case 6: return 0x1.bf78580000000p+0f;
      default: return 0.0f;
    }
  }
};

__device__ const float kCentroids4[16] = {
    -0x1.62013c0000000p+1f, -0x1.0cbd2c0000000p+1f, -0x1.a3e3b20000000p+0f, -0x1.46d1380000000p+0f,
    -0x1.eba5c80000000p-1f, -0x1.58a48e0000000p-1f, -0x1.9d829a0000000p-2f, -0x1.244e1e0000000p-3f,
    0x1.dfe6360000000p-4f, 0x1.842fb00000000p-2f, 0x1.4b8f4c0000000p-1f, 0x1.de181e0000000p-1f,
    0x1.40973a0000000p+0f, 0x1.9f2bd40000000p+0f, 0x1.09b21e0000000p+1f, 0x1.5c40d00000000p+1f,
};

struct LloydMax4 {
  static constexpr int kBits = 4;
  // decision boundary j (ascending), j = 0 .. 14
  __host__ __device__ static constexpr float boundary(int j) {
    switch (j) {
      case 0: return -0x1.375f340000000p+1f;
      case 1: return -0x1.deaf040000000p+0f;
      case 2: return -0x1.755a740000000p+0f;
      case 3: return -0x1.1e520e0000000p+0f;
      case 4: return -0x1.a2252c0000000p-1f;
      case 5: return -0x1.13b2ee0000000p-1f;
      case 6: return -0x1.17d4d40000000p-2f;
      case 7: return -0x1.a2d8180000000p-7f;
      case 8: return 0x1.fc293e0000000p-3f;
      case 9: return 0x1.06d3920000000p-1f;
      case 10: return 0x1.94d3b40000000p-1f;
      case 11: return 0x1.17d1a40000000p+0f;
      case 12: return 0x1.6fe1880000000p+0f;
      case 13: return 0x1.d948080000000p+0f;
      case 14: return 0x1.32f9780000000p+1f;
      default: return 0.0f;
    }
  }
};

__device__ const float kCentroids5[32] = {
    -0x1.ac91f60000000p+1f, -0x1.6321cc0000000p+1f, -0x1.3225e60000000p+1f, -0x1.0b561c0000000p+1f,
    -0x1.d699460000000p+0f, -0x1.a09a100000000p+0f, -0x1.6fd3ea0000000p+0f, -0x1.428b900000000p+0f,
    -0x1.188ad00000000p+0f, -0x1.e1e18a0000000p-1f, -0x1.9622100000000p-1f, -0x1.4d435a0000000p-1f,
    -0x1.05cbe20000000p-1f, -0x1.7eb07a0000000p-2f, -0x1.e608de0000000p-3f, -0x1.a506c60000000p-4f,
    0x1.0475740000000p-5f, 0x1.5047540000000p-3f, 0x1.334d940000000p-2f, 0x1.c2176e0000000p-2f,
    0x1.2961fa0000000p-1f, 0x1.7485660000000p-1f, 0x1.bf6f5e0000000p-1f, 0x1.0786a00000000p+0f,
    0x1.31bb120000000p+0f, 0x1.5f74700000000p+0f, 0x1.91513a0000000p+0f, 0x1.c764c40000000p+0f,
    0x1.02e1ba0000000p+1f, 0x1.279e360000000p+1f, 0x1.554b020000000p+1f, 0x1.9dd1400000000p+1f,
};

struct LloydMax5 {
  static constexpr int kBits = 5;
  // decision boundary j (ascending), j = 0 .. 30
  __host__ __device__ static constexpr float boundary(int j) {
    switch (j) {
      case 0: return -0x1.87d9e00000000p+1f;
      case 1: return -0x1.4aa3d80000000p+1f;
      case 2: return -0x1.1ebe000000000p+1f;
      case 3: return -0x1.f6a2c00000000p+0f;
      case 4: return -0x1.bb99ac0000000p+0f;
      case 5: return -0x1.8836fc0000000p+0f;
      case 6: return -0x1.592fbc0000000p+0f;
      case 7: return -0x1.2d8b300000000p+0f;
      case 8: return -0x1.04bdca0000000p+0f;
      case 9: return -0x1.bc01cc0000000p-1f;
      case 10: return -0x1.71b2b40000000p-1f;
      case 11: return -0x1.29879e0000000p-1f;
      case 12: return -0x1.c524200000000p-2f;
      case 13: return -0x1.38da740000000p-2f;
      case 14: return -0x1.5c46200000000p-3f;
      case 15: return -0x1.22cc0c0000000p-5f;
      case 16: return 0x1.9164b00000000p-4f;
      case 17: return 0x1.db713e0000000p-3f;
      case 18: return 0x1.7ab2800000000p-2f;
      case 19: return 0x1.0536d80000000p-1f;
      case 20: return 0x1.4ef3b00000000p-1f;
      case 21: return 0x1.99fa620000000p-1f;
      case 22: return 0x1.e73e500000000p-1f;
      case 23: return 0x1.1ca0d80000000p+0f;
      case 24: return 0x1.4897c00000000p+0f;
      case 25: return 0x1.7862d40000000p+0f;
      case 26: return 0x1.ac5b000000000p+0f;
      case 27: return 0x1.e6941c0000000p+0f;
      case 28: return 0x1.153ff80000000p+1f;
      case 29: return 0x1.3e749c0000000p+1f;
      case 30: return 0x1.798e200000000p+1f;
      default: return 0.0f;
    }
  }
};

__device__ const float kCentroids8[256] = {
    -0x1.205d0a0000000p+2f, -0x1.1d18780000000p+2f, -0x1.1bec1c0000000p+2f, -0x1.19b3a40000000p+2f,
    -0x1.173f520000000p+2f, -0x1.1542b80000000p+2f, -0x1.130a400000000p+2f, -0x1.10d1c80000000p+2f,
    -0x1.0e99520000000p+2f, -0x1.0c60dc0000000p+2f, -0x1.0a28640000000p+2f, -0x1.07efec0000000p+2f,
    -0x1.060b440000000p+2f, -0x1.02edb40000000p+2f, -0x1.002af20000000p+2f, -0x1.0023940000000p+2f,
    -0x1.f8a04e0000000p+1f, -0x1.f559c20000000p+1f, -0x1.f1731e0000000p+1f, -0x1.ec83300000000p+1f,
    -0x1.e641300000000p+1f, -0x1.e1a33e0000000p+1f, -0x1.df4c460000000p+1f, -0x1.da7dae0000000p+1f,
    -0x1.d65a000000000p+1f, -0x1.d0d4840000000p+1f, -0x1.cc295a0000000p+1f, -0x1.ca45dc0000000p+1f,
    -0x1.c51d2a0000000p+1f, -0x1.c07de60000000p+1f, -0x1.bbcbcc0000000p+1f, -0x1.b6ce2e0000000p+1f,
    -0x1.b2f5dc0000000p+1f, -0x1.ae7b260000000p+1f, -0x1.a9ea6e0000000p+1f, -0x1.a55f6a0000000p+1f,
    -0x1.a0ff200000000p+1f, -0x1.9c2c220000000p+1f, -0x1.98b3a00000000p+1f, -0x1.9420600000000p+1f,
    -0x1.8e4f8c0000000p+1f, -0x1.8a835e0000000p+1f, -0x1.867b620000000p+1f, -0x1.81e5540000000p+1f,
    -0x1.7d75d80000000p+1f, -0x1.7925520000000p+1f, -0x1.74a1e40000000p+1f, -0x1.6ff6de0000000p+1f,
    -0x1.6bad540000000p+1f, -0x1.672e5c0000000p+1f, -0x1.62c6a20000000p+1f, -0x1.5e69b60000000p+1f,
    -0x1.59f9580000000p+1f, -0x1.54ebce0000000p+1f, -0x1.50b0380000000p+1f, -0x1.4cc0480000000p+1f,
    -0x1.47cb880000000p+1f, -0x1.433c380000000p+1f, -0x1.3f541e0000000p+1f, -0x1.3b0e4e0000000p+1f,
    -0x1.3645f00000000p+1f, -0x1.31a27c0000000p+1f, -0x1.2cdda80000000p+1f, -0x1.287fc00000000p+1f,
    -0x1.2424dc0000000p+1f, -0x1.1f30040000000p+1f, -0x1.1ada980000000p+1f, -0x1.16aa080000000p+1f,
    -0x1.1286160000000p+1f, -0x1.0e415a0000000p+1f, -0x1.0a11fc0000000p+1f, -0x1.05b1fe0000000p+1f,
    -0x1.00d17a0000000p+1f, -0x1.f849600000000p+0f, -0x1.ee1af60000000p+0f, -0x1.e4a6ca0000000p+0f,
    -0x1.dbe5c40000000p+0f, -0x1.d23adc0000000p+0f, -0x1.c8edf80000000p+0f, -0x1.bf1dd00000000p+0f,
    -0x1.b5d8e20000000p+0f, -0x1.aca0360000000p+0f, -0x1.a3ae1c0000000p+0f, -0x1.9aa3220000000p+0f,
    -0x1.92215e0000000p+0f, -0x1.895b360000000p+0f, -0x1.80e9ba0000000p+0f, -0x1.781bdc0000000p+0f,
    -0x1.6f60760000000p+0f, -0x1.66f6a20000000p+0f, -0x1.5e70380000000p+0f, -0x1.55e92c0000000p+0f,
    -0x1.4d45b60000000p+0f, -0x1.4514060000000p+0f, -0x1.3c4bd80000000p+0f, -0x1.3381380000000p+0f,
    -0x1.2a9dbe0000000p+0f, -0x1.2168c60000000p+0f, -0x1.188f160000000p+0f, -0x1.0fba0e0000000p+0f,
    -0x1.0709ce0000000p+0f, -0x1.fcf1200000000p-1f, -0x1.ebfe860000000p-1f, -0x1.dad2420000000p-1f,
    -0x1.c92b460000000p-1f, -0x1.b7fc3c0000000p-1f, -0x1.a6fcce0000000p-1f, -0x1.9665a60000000p-1f,
    -0x1.8485240000000p-1f, -0x1.722d480000000p-1f, -0x1.5fcf780000000p-1f, -0x1.4db5660000000p-1f,
    -0x1.3b85560000000p-1f, -0x1.298cb00000000p-1f, -0x1.17b04a0000000p-1f, -0x1.05b2960000000p-1f,
    -0x1.e676680000000p-2f, -0x1.c1fe1a0000000p-2f, -0x1.9eb3b00000000p-2f, -0x1.7ab2000000000p-2f,
    -0x1.56283e0000000p-2f, -0x1.325f580000000p-2f, -0x1.0f010e0000000p-2f, -0x1.da7f980000000p-3f,
    -0x1.99e10a0000000p-3f, -0x1.5674b00000000p-3f, -0x1.12b6e80000000p-3f, -0x1.9af1c80000000p-4f,
    -0x1.0d2b820000000p-4f, -0x1.009b140000000p-5f, 0x1.1c9c8c0000000p-8f, 0x1.4abb300000000p-5f,
    0x1.3136b60000000p-4f, 0x1.b8caec0000000p-4f, 0x1.1f9c6a0000000p-3f, 0x1.64e6ec0000000p-3f,
    0x1.aa3f260000000p-3f, 0x1.f1c1440000000p-3f, 0x1.1ca4dc0000000p-2f, 0x1.42816e0000000p-2f,
    0x1.674e940000000p-2f, 0x1.8cbd0a0000000p-2f, 0x1.b06efc0000000p-2f, 0x1.d3d4600000000p-2f,
    0x1.f713060000000p-2f, 0x1.0d23c00000000p-1f, 0x1.1e03cc0000000p-1f, 0x1.2e9d280000000p-1f,
    0x1.3ffa220000000p-1f, 0x1.51a9460000000p-1f, 0x1.6379220000000p-1f, 0x1.74a86c0000000p-1f,
    0x1.8660a80000000p-1f, 0x1.97bfc60000000p-1f, 0x1.a9775c0000000p-1f, 0x1.ba98fa0000000p-1f,
    0x1.cbd49a0000000p-1f, 0x1.dd32520000000p-1f, 0x1.eee9640000000p-1f, 0x1.002dda0000000p+0f,
    0x1.08cd160000000p+0f, 0x1.116c9a0000000p+0f, 0x1.1a13880000000p+0f, 0x1.22b44c0000000p+0f,
    0x1.2bb3a80000000p+0f, 0x1.3430be0000000p+0f, 0x1.3d25b20000000p+0f, 0x1.4640ee0000000p+0f,
    0x1.4f69f20000000p+0f, 0x1.58182a0000000p+0f, 0x1.6081080000000p+0f, 0x1.68bf160000000p+0f,
    0x1.7145060000000p+0f, 0x1.7a1fc20000000p+0f, 0x1.83442c0000000p+0f, 0x1.8c57540000000p+0f,
    0x1.957ac80000000p+0f, 0x1.9e8bc40000000p+0f, 0x1.a7c84c0000000p+0f, 0x1.b145f80000000p+0f,
    0x1.ba317e0000000p+0f, 0x1.c30a340000000p+0f, 0x1.cc6ea20000000p+0f, 0x1.d5bff40000000p+0f,
    0x1.df06280000000p+0f, 0x1.e7fd2e0000000p+0f, 0x1.f1566c0000000p+0f, 0x1.fb0f4c0000000p+0f,
    0x1.021bb80000000p+1f, 0x1.065fdc0000000p+1f, 0x1.0ab4c40000000p+1f, 0x1.0f44d20000000p+1f,
    0x1.13eae40000000p+1f, 0x1.184b860000000p+1f, 0x1.1cc9f60000000p+1f, 0x1.20ee120000000p+1f,
    0x1.25ad800000000p+1f, 0x1.2a5a940000000p+1f, 0x1.2eab840000000p+1f, 0x1.32f5c00000000p+1f,
    0x1.3780a20000000p+1f, 0x1.3bcfb80000000p+1f, 0x1.406f480000000p+1f, 0x1.4493fc0000000p+1f,
    0x1.491dbc0000000p+1f, 0x1.4db1280000000p+1f, 0x1.51f6440000000p+1f, 0x1.56275c0000000p+1f,
    0x1.5acff20000000p+1f, 0x1.5f65860000000p+1f, 0x1.63c5540000000p+1f, 0x1.6843b80000000p+1f,
    0x1.6d084e0000000p+1f, 0x1.714fe80000000p+1f, 0x1.75b7d60000000p+1f, 0x1.7a3ccc0000000p+1f,
    0x1.7e68620000000p+1f, 0x1.82c03a0000000p+1f, 0x1.87e4720000000p+1f, 0x1.8d17160000000p+1f,
    0x1.929fc00000000p+1f, 0x1.9611be0000000p+1f, 0x1.9a441e0000000p+1f, 0x1.9e6fb60000000p+1f,
    0x1.a23c480000000p+1f, 0x1.a695e60000000p+1f, 0x1.aad1cc0000000p+1f, 0x1.af4ea40000000p+1f,
    0x1.b415060000000p+1f, 0x1.b894c60000000p+1f, 0x1.bb595c0000000p+1f, 0x1.c0515c0000000p+1f,
    0x1.c680f80000000p+1f, 0x1.c9976e0000000p+1f, 0x1.cd67b00000000p+1f, 0x1.d1f10a0000000p+1f,
    0x1.d8a98c0000000p+1f, 0x1.dbd2440000000p+1f, 0x1.dfd8be0000000p+1f, 0x1.e620580000000p+1f,
    0x1.e889f40000000p+1f, 0x1.eda4600000000p+1f, 0x1.f206ea0000000p+1f, 0x1.f5fb220000000p+1f,
    0x1.fcac3c0000000p+1f, 0x1.0093840000000p+2f, 0x1.01e5520000000p+2f, 0x1.0517880000000p+2f,
    0x1.06563e0000000p+2f, 0x1.088eb60000000p+2f, 0x1.0b0d9a0000000p+2f, 0x1.0cb27c0000000p+2f,
    0x1.0f381a0000000p+2f, 0x1.1170920000000p+2f, 0x1.13a90a0000000p+2f, 0x1.15e1800000000p+2f,
};

struct LloydMax8 {
  static constexpr int kBits = 8;
  // decision boundary j (ascending), j = 0 .. 254
  __host__ __device__ static constexpr float boundary(int j) {
    switch (j) {
      case 0: return -0x1.1ebac00000000p+2f;
      case 1: return -0x1.1c824a0000000p+2f;
      case 2: return -0x1.1acfe00000000p+2f;
      case 3: return -0x1.18797c0000000p+2f;
      case 4: return -0x1.1641040000000p+2f;
      case 5: return -0x1.14267c0000000p+2f;
      case 6: return -0x1.11ee040000000p+2f;
      case 7: return -0x1.0fb58c0000000p+2f;
      case 8: return -0x1.0d7d180000000p+2f;
      case 9: return -0x1.0b44a00000000p+2f;
      case 10: return -0x1.090c280000000p+2f;
      case 11: return -0x1.06fd980000000p+2f;
      case 12: return -0x1.047c7c0000000p+2f;
      case 13: return -0x1.018c540000000p+2f;
      case 14: return -0x1.0027440000000p+2f;
      case 15: return -0x1.fc73bc0000000p+1f;
      case 16: return -0x1.f6fd080000000p+1f;
      case 17: return -0x1.f366700000000p+1f;
      case 18: return -0x1.eefb280000000p+1f;
      case 19: return -0x1.e962300000000p+1f;
      case 20: return -0x1.e3f2380000000p+1f;
      case 21: return -0x1.e077c20000000p+1f;
      case 22: return -0x1.dce4fa0000000p+1f;
      case 23: return -0x1.d86bd80000000p+1f;
      case 24: return -0x1.d397420000000p+1f;
      case 25: return -0x1.ce7ef00000000p+1f;
      case 26: return -0x1.cb379c0000000p+1f;
      case 27: return -0x1.c7b1840000000p+1f;
      case 28: return -0x1.c2cd880000000p+1f;
      case 29: return -0x1.be24d80000000p+1f;
      case 30: return -0x1.b94cfc0000000p+1f;
      case 31: return -0x1.b4e2040000000p+1f;
      case 32: return -0x1.b0b8800000000p+1f;
      case 33: return -0x1.ac32ca0000000p+1f;
      case 34: return -0x1.a7a4ec0000000p+1f;
      case 35: return -0x1.a32f440000000p+1f;
      case 36: return -0x1.9e95a00000000p+1f;
      case 37: return -0x1.9a6fe00000000p+1f;
      case 38: return -0x1.966a000000000p+1f;
      case 39: return -0x1.9137f60000000p+1f;
      case 40: return -0x1.8c69740000000p+1f;
      case 41: return -0x1.887f600000000p+1f;
      case 42: return -0x1.84305c0000000p+1f;
      case 43: return -0x1.7fad960000000p+1f;
      case 44: return -0x1.7b4d940000000p+1f;
      case 45: return -0x1.76e39c0000000p+1f;
      case 46: return -0x1.724c600000000p+1f;
      case 47: return -0x1.6dd2180000000p+1f;
      case 48: return -0x1.696dd80000000p+1f;
      case 49: return -0x1.64fa800000000p+1f;
      case 50: return -0x1.60982c0000000p+1f;
      case 51: return -0x1.5c31880000000p+1f;
      case 52: return -0x1.5772940000000p+1f;
      case 53: return -0x1.52ce040000000p+1f;
      case 54: return -0x1.4eb8400000000p+1f;
      case 55: return -0x1.4a45e80000000p+1f;
      case 56: return -0x1.4583e00000000p+1f;
      case 57: return -0x1.41482c0000000p+1f;
      case 58: return -0x1.3d31360000000p+1f;
      case 59: return -0x1.38aa200000000p+1f;
      case 60: return -0x1.33f4360000000p+1f;
      case 61: return -0x1.2f40120000000p+1f;
      case 62: return -0x1.2aaeb40000000p+1f;
      case 63: return -0x1.26524e0000000p+1f;
      case 64: return -0x1.21aa700000000p+1f;
      case 65: return -0x1.1d054e0000000p+1f;
      case 66: return -0x1.18c2500000000p+1f;
      case 67: return -0x1.1498100000000p+1f;
      case 68: return -0x1.1063b80000000p+1f;
      case 69: return -0x1.0c29ac0000000p+1f;
      case 70: return -0x1.07e1fc0000000p+1f;
      case 71: return -0x1.0341bc0000000p+1f;
      case 72: return -0x1.fcf62a0000000p+0f;
      case 73: return -0x1.f3322c0000000p+0f;
      case 74: return -0x1.e960e00000000p+0f;
      case 75: return -0x1.e046480000000p+0f;
      case 76: return -0x1.d710500000000p+0f;
      case 77: return -0x1.cd946a0000000p+0f;
      case 78: return -0x1.c405e40000000p+0f;
      case 79: return -0x1.ba7b580000000p+0f;
      case 80: return -0x1.b13c8c0000000p+0f;
      case 81: return -0x1.a827280000000p+0f;
      case 82: return -0x1.9f28a00000000p+0f;
      case 83: return -0x1.9662400000000p+0f;
      case 84: return -0x1.8dbe4a0000000p+0f;
      case 85: return -0x1.8522780000000p+0f;
      case 86: return -0x1.7c82cc0000000p+0f;
      case 87: return -0x1.73be280000000p+0f;
      case 88: return -0x1.6b2b8c0000000p+0f;
      case 89: return -0x1.62b36c0000000p+0f;
      case 90: return -0x1.5a2cb20000000p+0f;
      case 91: return -0x1.5197700000000p+0f;
      case 92: return -0x1.492cde0000000p+0f;
      case 93: return -0x1.40aff00000000p+0f;
      case 94: return -0x1.37e6880000000p+0f;
      case 95: return -0x1.2f0f7c0000000p+0f;
      case 96: return -0x1.2603420000000p+0f;
      case 97: return -0x1.1cfbee0000000p+0f;
      case 98: return -0x1.1424920000000p+0f;
      case 99: return -0x1.0b61ee0000000p+0f;
      case 100: return -0x1.02c1300000000p+0f;
      case 101: return -0x1.f477d40000000p-1f;
      case 102: return -0x1.e368640000000p-1f;
      case 103: return -0x1.d1fec40000000p-1f;
      case 104: return -0x1.c093c00000000p-1f;
      case 105: return -0x1.af7c840000000p-1f;
      case 106: return -0x1.9eb13a0000000p-1f;
      case 107: return -0x1.8d75640000000p-1f;
      case 108: return -0x1.7b59360000000p-1f;
      case 109: return -0x1.68fe600000000p-1f;
      case 110: return -0x1.56c2700000000p-1f;
      case 111: return -0x1.449d5e0000000p-1f;
      case 112: return -0x1.3289040000000p-1f;
      case 113: return -0x1.209e7c0000000p-1f;
      case 114: return -0x1.0eb1700000000p-1f;
      case 115: return -0x1.f8edca0000000p-2f;
      case 116: return -0x1.d43a400000000p-2f;
      case 117: return -0x1.b058e40000000p-2f;
      case 118: return -0x1.8cb2d80000000p-2f;
      case 119: return -0x1.686d200000000p-2f;
      case 120: return -0x1.4443cc0000000p-2f;
      case 121: return -0x1.20b0340000000p-2f;
      case 122: return -0x1.fc40da0000000p-3f;
      case 123: return -0x1.ba30500000000p-3f;
      case 124: return -0x1.782adc0000000p-3f;
      case 125: return -0x1.3495cc0000000p-3f;
      case 126: return -0x1.e02fcc0000000p-4f;
      case 127: return -0x1.540ea40000000p-4f;
      case 128: return -0x1.8d790c0000000p-5f;
      case 129: return -0x1.ba0f040000000p-7f;
      case 130: return 0x1.6e4ec20000000p-6f;
      case 131: return 0x1.d6944e0000000p-5f;
      case 132: return 0x1.7500d00000000p-4f;
      case 133: return 0x1.fc01e00000000p-4f;
      case 134: return 0x1.4241ac0000000p-3f;
      case 135: return 0x1.8793080000000p-3f;
      case 136: return 0x1.ce00340000000p-3f;
      case 137: return 0x1.0ac2c00000000p-2f;
      case 138: return 0x1.2f93240000000p-2f;
      case 139: return 0x1.54e8000000000p-2f;
      case 140: return 0x1.7a05d00000000p-2f;
      case 141: return 0x1.9e96040000000p-2f;
      case 142: return 0x1.c221ae0000000p-2f;
      case 143: return 0x1.e573b40000000p-2f;
      case 144: return 0x1.0456a20000000p-1f;
      case 145: return 0x1.1593c60000000p-1f;
      case 146: return 0x1.26507a0000000p-1f;
      case 147: return 0x1.374ba40000000p-1f;
      case 148: return 0x1.48d1b40000000p-1f;
      case 149: return 0x1.5a91340000000p-1f;
      case 150: return 0x1.6c10c80000000p-1f;
      case 151: return 0x1.7d848a0000000p-1f;
      case 152: return 0x1.8f10380000000p-1f;
      case 153: return 0x1.a09b900000000p-1f;
      case 154: return 0x1.b2082c0000000p-1f;
      case 155: return 0x1.c336ca0000000p-1f;
      case 156: return 0x1.d483760000000p-1f;
      case 157: return 0x1.e60ddc0000000p-1f;
      case 158: return 0x1.f7a28c0000000p-1f;
      case 159: return 0x1.047d780000000p+0f;
      case 160: return 0x1.0d1cd80000000p+0f;
      case 161: return 0x1.15c0100000000p+0f;
      case 162: return 0x1.1e63ea0000000p+0f;
      case 163: return 0x1.2733fa0000000p+0f;
      case 164: return 0x1.2ff2340000000p+0f;
      case 165: return 0x1.38ab380000000p+0f;
      case 166: return 0x1.41b3500000000p+0f;
      case 167: return 0x1.4ad5700000000p+0f;
      case 168: return 0x1.53c10e0000000p+0f;
      case 169: return 0x1.5c4c980000000p+0f;
      case 170: return 0x1.64a0100000000p+0f;
      case 171: return 0x1.6d020e0000000p+0f;
      case 172: return 0x1.75b2640000000p+0f;
      case 173: return 0x1.7eb1f80000000p+0f;
      case 174: return 0x1.87cdc00000000p+0f;
      case 175: return 0x1.90e90e0000000p+0f;
      case 176: return 0x1.9a03460000000p+0f;
      case 177: return 0x1.a32a080000000p+0f;
      case 178: return 0x1.ac87220000000p+0f;
      case 179: return 0x1.b5bbbc0000000p+0f;
      case 180: return 0x1.be9dd80000000p+0f;
      case 181: return 0x1.c7bc6c0000000p+0f;
      case 182: return 0x1.d1174c0000000p+0f;
      case 183: return 0x1.da630e0000000p+0f;
      case 184: return 0x1.e381ac0000000p+0f;
      case 185: return 0x1.eca9cc0000000p+0f;
      case 186: return 0x1.f632dc0000000p+0f;
      case 187: return 0x1.ffa35e0000000p+0f;
      case 188: return 0x1.043dca0000000p+1f;
      case 189: return 0x1.088a500000000p+1f;
      case 190: return 0x1.0cfccc0000000p+1f;
      case 191: return 0x1.1197dc0000000p+1f;
      case 192: return 0x1.161b340000000p+1f;
      case 193: return 0x1.1a8abe0000000p+1f;
      case 194: return 0x1.1edc040000000p+1f;
      case 195: return 0x1.234dc80000000p+1f;
      case 196: return 0x1.28040a0000000p+1f;
      case 197: return 0x1.2c830c0000000p+1f;
      case 198: return 0x1.30d0a20000000p+1f;
      case 199: return 0x1.353b300000000p+1f;
      case 200: return 0x1.39a82c0000000p+1f;
      case 201: return 0x1.3e1f800000000p+1f;
      case 202: return 0x1.4281a20000000p+1f;
      case 203: return 0x1.46d8dc0000000p+1f;
      case 204: return 0x1.4b67720000000p+1f;
      case 205: return 0x1.4fd3b60000000p+1f;
      case 206: return 0x1.540ed00000000p+1f;
      case 207: return 0x1.587ba80000000p+1f;
      case 208: return 0x1.5d1abc0000000p+1f;
      case 209: return 0x1.61956c0000000p+1f;
      case 210: return 0x1.6604860000000p+1f;
      case 211: return 0x1.6aa6040000000p+1f;
      case 212: return 0x1.6f2c1c0000000p+1f;
      case 213: return 0x1.7383e00000000p+1f;
      case 214: return 0x1.77fa500000000p+1f;
      case 215: return 0x1.7c52980000000p+1f;
      case 216: return 0x1.80944e0000000p+1f;
      case 217: return 0x1.8552560000000p+1f;
      case 218: return 0x1.8a7dc40000000p+1f;
      case 219: return 0x1.8fdb6c0000000p+1f;
      case 220: return 0x1.9458c00000000p+1f;
      case 221: return 0x1.982aee0000000p+1f;
      case 222: return 0x1.9c59ea0000000p+1f;
      case 223: return 0x1.a056000000000p+1f;
      case 224: return 0x1.a469180000000p+1f;
      case 225: return 0x1.a8b3d80000000p+1f;
      case 226: return 0x1.ad10380000000p+1f;
      case 227: return 0x1.b1b1d40000000p+1f;
      case 228: return 0x1.b654e60000000p+1f;
      case 229: return 0x1.b9f7100000000p+1f;
      case 230: return 0x1.bdd55c0000000p+1f;
      case 231: return 0x1.c3692a0000000p+1f;
      case 232: return 0x1.c80c340000000p+1f;
      case 233: return 0x1.cb7f900000000p+1f;
      case 234: return 0x1.cfac5c0000000p+1f;
      case 235: return 0x1.d54d4c0000000p+1f;
      case 236: return 0x1.da3de80000000p+1f;
      case 237: return 0x1.ddd5800000000p+1f;
      case 238: return 0x1.e2fc8c0000000p+1f;
      case 239: return 0x1.e755260000000p+1f;
      case 240: return 0x1.eb172a0000000p+1f;
      case 241: return 0x1.efd5a40000000p+1f;
      case 242: return 0x1.f401060000000p+1f;
      case 243: return 0x1.f953b00000000p+1f;
      case 244: return 0x1.fee9a20000000p+1f;
      case 245: return 0x1.013c6c0000000p+2f;
      case 246: return 0x1.037e6c0000000p+2f;
      case 247: return 0x1.05b6e40000000p+2f;
      case 248: return 0x1.07727a0000000p+2f;
      case 249: return 0x1.09ce280000000p+2f;
      case 250: return 0x1.0be00c0000000p+2f;
      case 251: return 0x1.0df54c0000000p+2f;
      case 252: return 0x1.1054560000000p+2f;
      case 253: return 0x1.128cce0000000p+2f;
      case 254: return 0x1.14c5440000000p+2f;
      default: return 0.0f;
    }
  }
};

}  // namespace tq
