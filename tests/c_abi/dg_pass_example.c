/*
 * dg_pass_example.c -- one canvas pass through libdgcanvas.so from plain C (no Python): bf16
 * hidden states and vocabulary head made up from a seeded xorshift generator, the pass
 * (statistics, keep the K most confident slots, re-draw the rest), and everything written to a
 * file for checking.
 *
 *   dg_pass_example OUT B S V d K seed pass
 *
 * OUT receives, little-endian: int32 B, S, V, d, K, pass; uint64 seed; uint16 h bits [B*S*d];
 * uint16 w bits [V*d]; int32 canvas_in [B*S]; int32 canvas_out [B*S]; int32 argmax [B*S];
 * float conf [B*S]; float entropy [B*S]; uint8 kept [B*S]; float mean_entropy [B];
 * uint32 status. Exit status 0 when every call succeeded.
 */
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime.h>

#include "dgcanvas.h"

static uint64_t rng_state;

static uint64_t next_u64(void) {
    rng_state ^= rng_state << 13;
    rng_state ^= rng_state >> 7;
    rng_state ^= rng_state << 17;
    return rng_state;
}

/* uniform in [-1, 1) */
static float next_f(void) { return (float)((double)(next_u64() >> 11) * 0x1.0p-52 - 1.0); }

/* fp32 -> bf16 bits, round to nearest even (finite inputs) */
static uint16_t bf16_bits(float x) {
    uint32_t u;
    memcpy(&u, &x, 4);
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

#define CHECK_CUDA(call)                                                              \
    do {                                                                              \
        cudaError_t e_ = (call);                                                      \
        if (e_ != cudaSuccess) {                                                      \
            fprintf(stderr, "%s failed: %s\n", #call, cudaGetErrorString(e_));      \
            return 1;                                                                 \
        }                                                                             \
    } while (0)

int main(int argc, char** argv) {
    if (argc != 9) {
        fprintf(stderr, "usage: %s OUT B S V d K seed pass\n", argv[0]);
        return 2;
    }
    const int32_t B = atoi(argv[2]), S = atoi(argv[3]), V = atoi(argv[4]), d = atoi(argv[5]);
    const int32_t K = atoi(argv[6]);
    const uint64_t seed = strtoull(argv[7], NULL, 10);
    const int32_t pass = atoi(argv[8]);
    const size_t R = (size_t)B * S;

    rng_state = seed * 0x9E3779B97F4A7C15ull + 1;
    uint16_t* h = malloc(R * d * 2);
    uint16_t* w = malloc((size_t)V * d * 2);
    int32_t* canvas = malloc(R * 4);
    const float ws = 1.7320508f / 16.0f; /* w entries of standard deviation about 1/16 */
    for (size_t i = 0; i < R * d; ++i) h[i] = bf16_bits(2.0f * next_f());
    for (size_t i = 0; i < (size_t)V * d; ++i) w[i] = bf16_bits(ws * next_f());
    for (size_t i = 0; i < R; ++i) canvas[i] = (int32_t)(next_u64() % (uint64_t)V);

    void *dh, *dw, *dws;
    int32_t *dc_in, *dc_out, *darg;
    float *dconf, *dent, *dmean;
    uint8_t* dkept;
    uint32_t* dstatus;
    CHECK_CUDA(cudaMalloc(&dh, R * d * 2));
    CHECK_CUDA(cudaMalloc(&dw, (size_t)V * d * 2));
    CHECK_CUDA(cudaMalloc((void**)&dc_in, R * 4));
    CHECK_CUDA(cudaMalloc((void**)&dc_out, R * 4));
    CHECK_CUDA(cudaMalloc((void**)&darg, R * 4));
    CHECK_CUDA(cudaMalloc((void**)&dconf, R * 4));
    CHECK_CUDA(cudaMalloc((void**)&dent, R * 4));
    CHECK_CUDA(cudaMalloc((void**)&dkept, R));
    CHECK_CUDA(cudaMalloc((void**)&dmean, (size_t)B * 4));
    CHECK_CUDA(cudaMalloc((void**)&dstatus, 4));
    CHECK_CUDA(cudaMemcpy(dh, h, R * d * 2, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(dw, w, (size_t)V * d * 2, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(dc_in, canvas, R * 4, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemset(dstatus, 0, 4));

    dg_head_desc desc;
    memset(&desc, 0, sizeof(desc));
    desc.B = B;
    desc.S = S;
    desc.d = d;
    desc.V = V;
    desc.h_dtype = DG_BF16;
    desc.w_dtype = DG_BF16;
    desc.h = dh;
    desc.w = dw;
    desc.inv_temp = 1.0f;
    size_t ws_bytes = 0;
    int rc = dg_workspace_bytes(&desc, &ws_bytes);
    if (rc != DG_OK) {
        fprintf(stderr, "dg_workspace_bytes: %s\n", dg_status_string(rc));
        return 1;
    }
    CHECK_CUDA(cudaMalloc(&dws, ws_bytes)); /* cudaMalloc memory is 256-byte aligned */
    rc = dg_canvas_step(&desc, dc_in, dc_out, K, seed, (uint32_t)pass, darg, dconf, dent, dkept,
                        dmean, NULL, NULL, dws, ws_bytes, dstatus, NULL);
    if (rc != DG_OK) {
        fprintf(stderr, "dg_canvas_step: %s\n", dg_status_string(rc));
        return 1;
    }
    CHECK_CUDA(cudaDeviceSynchronize());

    int32_t* c_out = malloc(R * 4);
    int32_t* arg = malloc(R * 4);
    float* conf = malloc(R * 4);
    float* ent = malloc(R * 4);
    uint8_t* kept = malloc(R);
    float* mean = malloc((size_t)B * 4);
    uint32_t status = 0;
    CHECK_CUDA(cudaMemcpy(c_out, dc_out, R * 4, cudaMemcpyDeviceToHost));
    CHECK_CUDA(cudaMemcpy(arg, darg, R * 4, cudaMemcpyDeviceToHost));
    CHECK_CUDA(cudaMemcpy(conf, dconf, R * 4, cudaMemcpyDeviceToHost));
    CHECK_CUDA(cudaMemcpy(ent, dent, R * 4, cudaMemcpyDeviceToHost));
    CHECK_CUDA(cudaMemcpy(kept, dkept, R, cudaMemcpyDeviceToHost));
    CHECK_CUDA(cudaMemcpy(mean, dmean, (size_t)B * 4, cudaMemcpyDeviceToHost));
    CHECK_CUDA(cudaMemcpy(&status, dstatus, 4, cudaMemcpyDeviceToHost));

    FILE* f = fopen(argv[1], "wb");
    if (!f) {
        perror("fopen");
        return 1;
    }
    const int32_t hdr[6] = {B, S, V, d, K, pass};
    fwrite(hdr, 4, 6, f);
    fwrite(&seed, 8, 1, f);
    fwrite(h, 2, R * d, f);
    fwrite(w, 2, (size_t)V * d, f);
    fwrite(canvas, 4, R, f);
    fwrite(c_out, 4, R, f);
    fwrite(arg, 4, R, f);
    fwrite(conf, 4, R, f);
    fwrite(ent, 4, R, f);
    fwrite(kept, 1, R, f);
    fwrite(mean, 4, (size_t)B, f);
    fwrite(&status, 4, 1, f);
    fclose(f);
    printf("pass done: status %u, mean entropy of canvas 0 %.6f nats\n", status, mean[0]);
    return status == 0 ? 0 : 1;
}
