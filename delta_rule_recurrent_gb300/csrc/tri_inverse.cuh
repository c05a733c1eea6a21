// tri_inverse.cuh -- (I + A)^{-1} for a strictly lower-triangular 64 x 64 A.
//
// The chunk form needs T = (I + A)^{-1} diag(beta) with
// A = tril(diag(beta) K K^T, -1); the pages compute the triangular inverse by
// forward substitution rather than a dense inverse ("Hardware-efficient
// implementation", section 3 of paperlayer.ai/abs/2406.06484v6; "Restauration
// de la dépendance causale", fr.news.hada.io/topic?id=31925, which also notes
// the blocks of 16 tokens used in practice).
#pragma once

namespace dn {

constexpr int kTriPitch = 65;  // default row pitch (floats) of the 64 x 64 operands

// A and X are 64 x 64 fp32 in shared memory with row pitch L; Ys is
// 3 x 16 x 17 floats of scratch.  The four 16 x 16 diagonal blocks are
// inverted by column-wise substitution, then the block diagonals below them
// follow from X_ij = -X_ii * sum_{l=j}^{i-1} A_il X_lj.  All NT threads of the
// block must call it; it ends with a barrier.
template <int NT, int L = kTriPitch>
__device__ void unit_lower_inverse64(const float* __restrict__ Am, float* __restrict__ Xm,
                                     float* __restrict__ Ys) {
    const int tid = threadIdx.x;
    if (tid < 64) {
        const int base = (tid >> 4) * 16, c = tid & 15;
        float x[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            float acc = (r == c) ? 1.f : 0.f;
#pragma unroll
            for (int l = 0; l < r; ++l) acc = fmaf(-Am[(base + r) * L + base + l], x[l], acc);
            x[r] = (r < c) ? 0.f : acc;
            Xm[(base + r) * L + base + c] = x[r];
        }
    }
    // Blocks above the diagonal are zero: (0,1) (0,2) (0,3) (1,2) (1,3) (2,3).
    for (int e = tid; e < 6 * 256; e += NT) {
        const int blk = e >> 8, r = (e >> 4) & 15, c = e & 15;
        const int bi = blk < 3 ? 0 : (blk < 5 ? 1 : 2);
        const int bj = blk < 3 ? blk + 1 : (blk < 5 ? blk - 1 : 3);
        Xm[(16 * bi + r) * L + 16 * bj + c] = 0.f;
    }
    __syncthreads();
    for (int d = 1; d < 4; ++d) {
        const int nb = 4 - d;
        for (int e = tid; e < nb * 256; e += NT) {
            const int j = e >> 8, r = (e >> 4) & 15, c = e & 15, i = j + d;
            float acc = 0.f;
            for (int kk = 16 * j; kk < 16 * i; ++kk)
                acc = fmaf(Am[(16 * i + r) * L + kk], Xm[kk * L + 16 * j + c], acc);
            Ys[j * 272 + r * 17 + c] = acc;
        }
        __syncthreads();
        for (int e = tid; e < nb * 256; e += NT) {
            const int j = e >> 8, r = (e >> 4) & 15, c = e & 15, i = j + d;
            float acc = 0.f;
            for (int m = 0; m <= r; ++m)
                acc = fmaf(Xm[(16 * i + r) * L + 16 * i + m], Ys[j * 272 + m * 17 + c], acc);
            Xm[(16 * i + r) * L + 16 * j + c] = -acc;
        }
        __syncthreads();
    }
}

}  // namespace dn
