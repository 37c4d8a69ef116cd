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
