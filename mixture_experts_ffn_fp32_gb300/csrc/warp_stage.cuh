// Warp-wide moves of a 32-row x 64-byte block between registers (row `lane`
// in this lane's four 16-byte chunks) and row-major global memory, through a
// 2 KB per-warp staging buffer in shared memory: 16-byte chunks are
// XOR-swizzled by row, so both the row-wise and the column-wise shared
// accesses are bank-conflict free, and every global access instruction moves
// 8 rows x 64 contiguous bytes.
#pragma once

#include "common.cuh"

namespace moe {

// Stores the block; rows >= valid_rows and 16-byte chunks >= valid_chunks are
// not written.
MOE_DEV void warp_store_block(uint4* stg, const uint4 (&v)[4], int lane, char* row0,
                              size_t pitch, int valid_rows, int valid_chunks) {
    const int sw = (lane >> 1) & 3;
#pragma unroll
    for (int c = 0; c < 4; ++c) stg[lane * 4 + (c ^ sw)] = v[c];
    __syncwarp();
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int row = 8 * i + (lane >> 2);
        const int ch = lane & 3;
        const uint4 w = stg[row * 4 + (ch ^ ((row >> 1) & 3))];
        if (row < valid_rows && ch < valid_chunks)
            *reinterpret_cast<uint4*>(row0 + row * pitch + ch * 16) = w;
    }
    __syncwarp();
}

// The global half of warp_store_block, for a block already in the staging
// buffer in its swizzled layout (chunk c of row r at 16-byte slot
// r * 4 + (c ^ ((r >> 1) & 3))).
MOE_DEV void warp_flush_block(const uint4* stg, int lane, char* row0, size_t pitch, int valid_rows,
                              int valid_chunks) {
    __syncwarp();
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int row = 8 * i + (lane >> 2);
        const int ch = lane & 3;
        const uint4 w = stg[row * 4 + (ch ^ ((row >> 1) & 3))];
        if (row < valid_rows && ch < valid_chunks)
            *reinterpret_cast<uint4*>(row0 + row * pitch + ch * 16) = w;
    }
    __syncwarp();
}

// Column `lane` of a 32-row x 32-column BF16 block into the staging buffer in
// warp_flush_block's layout: v[i] is row i.
MOE_DEV void warp_stage_bf16_column(uint4* stg, int lane, const float (&v)[32]) {
    unsigned short* b = reinterpret_cast<unsigned short*>(stg);
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        const __nv_bfloat16 h = __float2bfloat16_rn(v[i]);
        b[(i * 4 + ((lane >> 3) ^ ((i >> 1) & 3))) * 8 + (lane & 7)] = *reinterpret_cast<const unsigned short*>(&h);
    }
}

// A 16-row x 32-column FP32 block, column `lane` from v (v[i] is row i),
// stored row-major (128 bytes per row) from the staging buffer: every store
// instruction moves 4 rows x 128 contiguous bytes. Rows >= valid_rows and
// 16-byte chunks >= valid_chunks are not written.
MOE_DEV void warp_store_f32_columns(uint4* stg, int lane, const float (&v)[16], char* row0, size_t pitch,
                                    int valid_rows, int valid_chunks) {
    float* f = reinterpret_cast<float*>(stg);
#pragma unroll
    for (int i = 0; i < 16; ++i) f[i * 32 + lane] = v[i];
    __syncwarp();
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int idx = lane + 32 * k;
        const int row = idx >> 3, ch = idx & 7;
        const uint4 w = stg[idx];
        if (row < valid_rows && ch < valid_chunks)
            *reinterpret_cast<uint4*>(row0 + row * pitch + ch * 16) = w;
    }
    __syncwarp();
}

// The same 16 x 32 block in the 24-bit blocked layout (f32_to_f24): per row,
// 32 16-bit high parts at hi_off and 32 8-bit low parts at lo_off (byte
// offsets from the row's start); rows >= valid_rows are not written.
MOE_DEV void warp_store_f24_columns(uint4* stg, int lane, const float (&v)[16], char* row0, size_t pitch,
                                    int valid_rows, size_t hi_off, size_t lo_off) {
    unsigned short* h = reinterpret_cast<unsigned short*>(stg);          // [16][32], 1 KB
    unsigned char* l = reinterpret_cast<unsigned char*>(stg) + 1024;     // [16][32], 512 bytes
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const uint32_t f = f32_to_f24(v[i]);
        h[i * 32 + lane] = static_cast<unsigned short>(f >> 8);
        l[i * 32 + lane] = static_cast<unsigned char>(f & 0xFFu);
    }
    __syncwarp();
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const int idx = lane + 32 * k, row = idx >> 2, ch = idx & 3;
        if (row < valid_rows)
            *reinterpret_cast<uint4*>(row0 + row * pitch + hi_off + ch * 16) = stg[idx];
    }
    {
        const int row = lane >> 1, ch = lane & 1;
        if (row < valid_rows)
            *reinterpret_cast<uint4*>(row0 + row * pitch + lo_off + ch * 16) = stg[64 + lane];
    }
    __syncwarp();
}

// Loads the block in two steps, so that the global loads can be in flight
// while other work runs: warp_load_issue reads it row-major (rows >=
// valid_rows as zeros) into w, warp_load_finish turns w into the lane = row
// layout through the staging buffer.
MOE_DEV void warp_load_issue(uint4 (&w)[4], int lane, const char* row0, size_t pitch, int valid_rows) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int row = 8 * i + (lane >> 2);
        w[i] = make_uint4(0u, 0u, 0u, 0u);
        if (row < valid_rows) w[i] = *reinterpret_cast<const uint4*>(row0 + row * pitch + (lane & 3) * 16);
    }
}

MOE_DEV void warp_load_finish(uint4* stg, const uint4 (&w)[4], uint4 (&v)[4], int lane) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int row = 8 * i + (lane >> 2);
        stg[row * 4 + ((lane & 3) ^ ((row >> 1) & 3))] = w[i];
    }
    __syncwarp();
    const int sw = (lane >> 1) & 3;
#pragma unroll
    for (int c = 0; c < 4; ++c) v[c] = stg[lane * 4 + (c ^ sw)];
    __syncwarp();
}

}  // namespace moe
