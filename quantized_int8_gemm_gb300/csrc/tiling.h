// tiling.h -- the pre-tiled operand planes the GEMM streams with 1-D bulk
// copies, defined once for their producers (registration, activation
// prepass) and their consumer (the GEMM kernel).
//
// The GEMM runs 128 (tokens) x 128 (weight rows) output tiles over K in
// stages of 128; two stages make one 256-element super-block.  Every
// (tile, super-block, half) owns one contiguous block in global memory laid
// out exactly as the kernel's shared-memory stage buffer, so one bulk copy
// per operand per stage moves it.
//
// Operand image (both A and B): two K-blocks of 64 fp16 (k = 0..63, 64..127
// of the stage), each 128 rows x 128 B with the 128-byte swizzle that UMMA's
// SWIZZLE_128B descriptor expects: row r of a K-block at (r/8)*1024 + (r%8)*128,
// its 16-byte chunk j stored at chunk position j ^ (r%8).
//
// Min-term image (q4_K, odd half only): 128 rows x 16 fp16 (32 B per row)
// with the 32-byte swizzle (SWIZZLE_32B descriptor): row r at
// (r/8)*256 + (r%8)*32, 16-byte chunk j stored at j ^ ((r%8)/4).
//   A side: slot 2c = hi(g'), slot 2c+1 = lo(g') of 32-chunk c of the super-block
//   B side: slots 2c and 2c+1 both = m (the 6-bit min of sub-block c)
//
// Block layouts (byte offsets inside one block):
//   A even: [operand 32768]
//   A odd : [operand 32768][q4_K: A min 4096]
//   B even: [operand 32768]
//   B odd : [operand 32768][q4_K: B min 4096]
// Blocks of one tile are ordered (super-block, half).
//
// The weight plane ends with a scale region: per (weight tile, super-block)
// one scale block [d 128 x f32][q4_K: dmin 128 x f32], ordered like the
// operand pairs.  The GEMM's epilogue reads it through its own small ring,
// so the operand stages are freed by the tensor core alone.
#pragma once
#include <cstdint>

namespace mmq {
namespace tiling {

constexpr int kTileM = 128;  // tokens per tile
constexpr int kTileN = 128;  // weight rows per tile
constexpr int kStageK = 128;
constexpr int kOperandBytes = kTileM * kStageK * 2;  // 32768 (kTileM == kTileN)
constexpr int kMinBytes = 128 * 32;                  // 4096
constexpr int kScaleBytes = kTileN * 4;              // 512

__host__ __device__ constexpr int a_even_bytes() { return kOperandBytes; }
__host__ __device__ constexpr int a_odd_bytes(bool q4) { return kOperandBytes + (q4 ? kMinBytes : 0); }
__host__ __device__ constexpr int b_even_bytes() { return kOperandBytes; }
__host__ __device__ constexpr int b_odd_bytes(bool q4) { return kOperandBytes + (q4 ? kMinBytes : 0); }
__host__ __device__ constexpr int a_pair_bytes(bool q4) { return a_even_bytes() + a_odd_bytes(q4); }
__host__ __device__ constexpr int b_pair_bytes(bool q4) { return b_even_bytes() + b_odd_bytes(q4); }
// one scale block: d (and dmin for q4_K) of the 128 rows of a weight tile
__host__ __device__ constexpr int scale_block_bytes(bool q4) { return kScaleBytes * (q4 ? 2 : 1); }

constexpr int kAMin = kOperandBytes;   // A min image in an odd A block (q4_K)
constexpr int kBMin = kOperandBytes;   // B min image in an odd B block (q4_K)
constexpr int kSDmin = kScaleBytes;    // dmin row in a scale block (q4_K)

// byte offset of element (row, k) of a stage operand image, k in [0, 128)
__host__ __device__ constexpr uint32_t operand_off(int row, int k) {
  return static_cast<uint32_t>((k >> 6) * 16384 + (row >> 3) * 1024 + (row & 7) * 128 +
                               ((((k & 63) >> 3) ^ (row & 7)) << 4) + (k & 7) * 2);
}
// byte offset of slot j in [0,16) of row r in a min-term image
__host__ __device__ constexpr uint32_t min_off(int row, int j) {
  return static_cast<uint32_t>((row >> 3) * 256 + (row & 7) * 32 +
                               (((j >> 3) ^ ((row & 7) >> 2)) << 4) + (j & 7) * 2);
}
// first byte of block (tile, sb, half) in a plane of `nsb` super-blocks per tile
__host__ __device__ constexpr uint64_t a_block(int64_t tile, int64_t sb, int half, int64_t nsb,
                                               bool q4) {
  return static_cast<uint64_t>((tile * nsb + sb) * a_pair_bytes(q4) + (half ? a_even_bytes() : 0));
}
__host__ __device__ constexpr uint64_t b_block(int64_t tile, int64_t sb, int half, int64_t nsb,
                                               bool q4) {
  return static_cast<uint64_t>((tile * nsb + sb) * b_pair_bytes(q4) + (half ? b_even_bytes() : 0));
}
// first byte of the scale region of a weight plane with n_ot tiles
__host__ __device__ constexpr uint64_t b_scale_region(int64_t n_ot, int64_t nsb, bool q4) {
  return static_cast<uint64_t>(n_ot * nsb) * b_pair_bytes(q4);
}
// scale block (tile, sb), relative to the scale region
__host__ __device__ constexpr uint64_t b_scale_block(int64_t tile, int64_t sb, int64_t nsb, bool q4) {
  return static_cast<uint64_t>((tile * nsb + sb) * scale_block_bytes(q4));
}

// ---------------------------------------------------------------- split arm
// The split arm folds the activation scale into the A operand: each element
// a = da' * qs (exact in fp32) travels as fp16 hi = rn(a) and lo = rn(a - hi).
// Its activation block per (token tile, super-block, half) holds, per 64-K
// quarter kb of the half, the hi and lo K-blocks side by side, so one 64-K
// GEMM stage is one contiguous copy:
//   [hi kb0 16384][lo kb0 16384][hi kb1 16384][lo kb1 16384][odd, q4_K: A min 4096]
// (a K-block: 128 rows x 128 B with the 128-byte swizzle, as above).  The
// weight side is the registered operand plane, unchanged.
constexpr int kSplitQuarter = 2 * kTileM * 64 * 2;  // 32768: hi + lo of one 64-K quarter
constexpr int kSplitLo = kTileM * 64 * 2;           // 16384: lo K-block after its hi
constexpr int kSplitMin = 2 * kSplitQuarter;        // A min image in an odd split block (q4_K)
__host__ __device__ constexpr int as_even_bytes() { return 2 * kSplitQuarter; }
__host__ __device__ constexpr int as_odd_bytes(bool q4) { return 2 * kSplitQuarter + (q4 ? kMinBytes : 0); }
__host__ __device__ constexpr int as_pair_bytes(bool q4) { return as_even_bytes() + as_odd_bytes(q4); }
__host__ __device__ constexpr uint64_t as_block(int64_t tile, int64_t sb, int half, int64_t nsb, bool q4) {
  return static_cast<uint64_t>((tile * nsb + sb) * as_pair_bytes(q4) + (half ? as_even_bytes() : 0));
}
// byte offset of the hi element (row, k), k in [0, 128), inside a split block
__host__ __device__ constexpr uint32_t split_off(int row, int k) {
  return static_cast<uint32_t>((k >> 6) * kSplitQuarter) + operand_off(row, k & 63);
}

// ---------------------------------------------------------------- pair arm
// The pair arm's activation plane: token tiles of TP = 2H rows (H a multiple
// of 8, at most 64), one block per (token tile, super-block, half) holding the
// hi and lo images grouped by the H-row half of the tile that one CTA of an SM
// pair stages, so that a CTA's share of a half super-block is one contiguous
// copy:
//   [rows 0..H-1:  hi kb0][lo kb0][hi kb1][lo kb1][odd, q4_K: A min]
//   [rows H..2H-1: the same]
// (an H-row K-block: H rows x 128 B with the 128-byte swizzle, H * 128 bytes;
// the min image H rows x 16 slots with the 32-byte swizzle, H * 32 bytes).
// With H = 64 a block holds the split arm's bytes, regrouped.
__host__ __device__ constexpr int pair_kb_bytes(int h) { return h * 128; }
__host__ __device__ constexpr int pair_rank_bytes(bool q4, int half, int h) {
  return 4 * pair_kb_bytes(h) + (q4 && half ? h * 32 : 0);
}
// bytes of one (token tile, super-block): its even and its odd block
__host__ __device__ constexpr int pair_sb_bytes(bool q4, int h) {
  return 2 * pair_rank_bytes(q4, 0, h) + 2 * pair_rank_bytes(q4, 1, h);
}
__host__ __device__ constexpr uint64_t pair_block(int64_t tile, int64_t sb, int half, int64_t nsb, bool q4, int h) {
  return static_cast<uint64_t>((tile * nsb + sb) * pair_sb_bytes(q4, h) + (half ? 2 * pair_rank_bytes(q4, 0, h) : 0));
}
// byte offset of the hi element (row, k), row in [0, 2h), k in [0, 128), inside
// a pair block; its lo element is pair_kb_bytes(h) further
__host__ __device__ constexpr uint32_t pair_off(int row, int k, bool q4, int half, int h) {
  return static_cast<uint32_t>((row / h) * pair_rank_bytes(q4, half, h) + (k >> 6) * 2 * pair_kb_bytes(h)) +
         operand_off(row % h, k & 63);
}
// byte offset of min-term slot j of row r inside an odd pair block (q4_K)
__host__ __device__ constexpr uint32_t pair_min_off(int row, int j, int h) {
  return static_cast<uint32_t>((row / h) * pair_rank_bytes(true, 1, h) + 4 * pair_kb_bytes(h)) + min_off(row % h, j);
}

// ---------------------------------------------------------------- raw plane
// The raw arm streams the packed weight bytes and unpacks them in the GEMM.
// Per (weight tile, super-block, half) one raw block holds the bytes of that
// half of the 128 rows' k-quant blocks, regrouped so that a converter thread
// (one row) and its neighbours (the next rows) read consecutive 8-byte words:
//   q4_K: qs   [g = kb*4 + j][row] 8 B: qs bytes 32*kb + 8*j .. +7 of the half
//                (low nibbles: k = 64*kb + 8*j .., high nibbles: k + 32 ..)
//         sc   [sub 0..3][row] fp16: the 6-bit scale of sub-block 4*half+sub
//   q6_K: ql   [j 0..7][row] 8 B: ql bytes 8*j .. +7 of the half
//                (low nibbles: k = 8*j .., high nibbles: k = 64 + 8*j ..)
//         qh   [j 0..3][row] 8 B: qh bytes 8*j .. +7 of the half
//                (bit pair 2*p is k = 32*p + 8*j ..)
//         sc   [sub 0..7][row] fp16: the int8 scale of 16-element sub-block
//                8*half + sub
// where the half's bytes are q4_K qs[64*half ..], q6_K ql[64*half ..] and
// qh[32*half ..].  The scale region (d, dmin) and, for q4_K, the B min
// images are read from the operand plane, which the raw arm otherwise skips.
constexpr int kRawQ4Qs = 0, kRawQ4Sc = 8192, kRawQ4Bytes = 8192 + 1024;
constexpr int kRawQ6Ql = 0, kRawQ6Qh = 8192, kRawQ6Sc = 8192 + 4096, kRawQ6Bytes = 8192 + 4096 + 2048;
__host__ __device__ constexpr int raw_block_bytes(bool q4) { return q4 ? kRawQ4Bytes : kRawQ6Bytes; }
__host__ __device__ constexpr uint64_t raw_block(int64_t tile, int64_t sb, int half, int64_t nsb, bool q4) {
  return static_cast<uint64_t>(((tile * nsb + sb) * 2 + half) * raw_block_bytes(q4));
}

}  // namespace tiling
}  // namespace mmq
