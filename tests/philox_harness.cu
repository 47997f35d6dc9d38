// Device check of the library's Philox4x32-10 (fa_philox in csrc/fa_internal.cuh) against the
// published known-answer vectors (Salmon, Moraes, Dror, Shaw, SC'11; the vectors distributed
// with the generator's reference release, stored in tests/golden/philox4x32_10_kat.txt).
// Reads lines "c0 c1 c2 c3 k0 k1 -> o0 o1 o2 o3" (hex) from the file, runs one GPU thread per
// vector through the library's device function, and prints "ok N" or the first mismatch;
// exits non-zero on a mismatch or a CUDA error.
#include <cstdio>
#include <cstring>
#include <vector>

#include "../constrained_decoding_diffusion_gb300/csrc/fa_internal.cuh"

__global__ void k_philox(const uint32_t *in, uint32_t *out, int n) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    const uint32_t *c = in + 6 * i;
    const fa_u4 r = fa_philox(c[0], c[1], c[2], c[3], c[4], c[5]);
    out[4 * i + 0] = r.x;
    out[4 * i + 1] = r.y;
    out[4 * i + 2] = r.z;
    out[4 * i + 3] = r.w;
}

int main(int argc, char **argv) {
    if (argc < 2) return 2;
    FILE *f = fopen(argv[1], "r");
    if (!f) return 2;
    std::vector<uint32_t> in, want;
    char line[512];
    while (fgets(line, sizeof line, f)) {
        if (line[0] == '#' || strlen(line) < 10) continue;
        unsigned v[10];
        if (sscanf(line, "%x %x %x %x %x %x %x %x %x %x", &v[0], &v[1], &v[2], &v[3], &v[4], &v[5], &v[6], &v[7],
                   &v[8], &v[9]) != 10)
            return 2;
        for (int j = 0; j < 6; ++j) in.push_back(v[j]);
        for (int j = 6; j < 10; ++j) want.push_back(v[j]);
    }
    fclose(f);
    const int n = (int)(in.size() / 6);
    if (n == 0) return 2;
    uint32_t *d_in = nullptr, *d_out = nullptr;
    if (cudaMalloc(&d_in, in.size() * 4) != cudaSuccess || cudaMalloc(&d_out, want.size() * 4) != cudaSuccess) return 3;
    cudaMemcpy(d_in, in.data(), in.size() * 4, cudaMemcpyHostToDevice);
    k_philox<<<1, 32>>>(d_in, d_out, n);
    std::vector<uint32_t> got(want.size());
    if (cudaMemcpy(got.data(), d_out, got.size() * 4, cudaMemcpyDeviceToHost) != cudaSuccess) return 3;
    cudaFree(d_in);
    cudaFree(d_out);
    for (int i = 0; i < n; ++i)
        for (int j = 0; j < 4; ++j)
            if (got[4 * i + j] != want[4 * i + j]) {
                printf("mismatch vector %d word %d: got %08x want %08x\n", i, j, got[4 * i + j], want[4 * i + j]);
                return 1;
            }
    printf("ok %d\n", n);
    return 0;
}
