/*
 * Black-box run of cuRAND's device-API Philox4_32_10 generator (no source of
 * it is read or copied; it is only called).  For each record (seed, layer,
 * draw, token, j) the generator is initialised with
 *   subsequence = draw + layer * 2^32,  offset = 4 (j + token * 2^32)
 * and its first four words are written out.  The test that builds this
 * program compares them with the oracle's Philox4x32-10 of the counter
 * (j, token, draw, layer): subsequence and offset address the counter's high
 * and low 64 bits, so the fourth counter word (the layer) is exercised.
 *
 *   usage: curand_device_philox <records.bin> <words.bin>
 */
#include <curand_kernel.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>

typedef struct {
    unsigned long long seed;
    unsigned int layer, draw, token, j;
} Rec;

__global__ void first_words(const Rec* r, int n, uint4* out) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    curandStatePhilox4_32_10_t st;
    const unsigned long long sub = (unsigned long long)r[i].draw |
                                   ((unsigned long long)r[i].layer << 32);
    const unsigned long long off = 4ull * ((unsigned long long)r[i].j |
                                           ((unsigned long long)r[i].token << 32));
    curand_init(r[i].seed, sub, off, &st);
    out[i] = curand4(&st);
}

int main(int argc, char** argv) {
    if (argc != 3) return 2;
    FILE* f = fopen(argv[1], "rb");
    if (!f) return 3;
    fseek(f, 0, SEEK_END);
    const long bytes = ftell(f);
    fseek(f, 0, SEEK_SET);
    const int n = (int)(bytes / sizeof(Rec));
    Rec* h = (Rec*)malloc(sizeof(Rec) * (n > 0 ? n : 1));
    if (fread(h, sizeof(Rec), n, f) != (size_t)n) return 4;
    fclose(f);
    Rec* d;
    uint4* o;
    if (cudaMalloc(&d, sizeof(Rec) * n) != cudaSuccess) return 5;
    if (cudaMalloc(&o, sizeof(uint4) * n) != cudaSuccess) return 5;
    cudaMemcpy(d, h, sizeof(Rec) * n, cudaMemcpyHostToDevice);
    first_words<<<(n + 127) / 128, 128>>>(d, n, o);
    uint4* ho = (uint4*)malloc(sizeof(uint4) * n);
    if (cudaMemcpy(ho, o, sizeof(uint4) * n, cudaMemcpyDeviceToHost) != cudaSuccess) return 6;
    FILE* g = fopen(argv[2], "wb");
    if (!g) return 7;
    fwrite(ho, sizeof(uint4), n, g);
    fclose(g);
    cudaFree(d);
    cudaFree(o);
    free(h);
    free(ho);
    return 0;
}
