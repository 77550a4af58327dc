"""The C ABI from C: a small C program, compiled with gcc against
include/ws.h and linked with libws.so and the CUDA runtime, allocates device
memory itself, runs ws_preprocess and ws_topk (a short-row batch and a long
row that needs a workspace) and writes the results to files.  No Python
sits between the program and the library; the results must equal the
oracle's (preprocess within 1e-5, Top-K bit-exact)."""
import os
import subprocess

import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CLIENT = r"""
#include <stdio.h>
#include <stdlib.h>
#include <cuda_runtime.h>
#include "ws.h"

#define CHECK_WS(call) do { ws_status s_ = (call); if (s_ != WS_OK) { \
    fprintf(stderr, "%s: %s (%s)\n", #call, ws_status_string(s_), ws_last_error()); return 1; } } while (0)
#define CHECK_CUDA(call) do { cudaError_t e_ = (call); if (e_ != cudaSuccess) { \
    fprintf(stderr, "%s: %s\n", #call, cudaGetErrorString(e_)); return 1; } } while (0)

static void* slurp(const char* path, size_t bytes) {
    void* p = malloc(bytes);
    FILE* f = fopen(path, "rb");
    if (!p || !f || fread(p, 1, bytes, f) != bytes) { fprintf(stderr, "cannot read %s\n", path); exit(1); }
    fclose(f);
    return p;
}

static void dump(const char* path, const void* p, size_t bytes) {
    FILE* f = fopen(path, "wb");
    if (!f || fwrite(p, 1, bytes, f) != bytes) { fprintf(stderr, "cannot write %s\n", path); exit(1); }
    fclose(f);
}

int main(int argc, char** argv) {
    if (argc != 2) return 2;
    const char* dir = argv[1];
    char path[4096];
    enum { B = 3, SW = 320, SH = 180, DW = 96, DH = 96, R1 = 4, C1 = 1000, K1 = 5, R2 = 2, C2 = 50000, K2 = 32 };
    const size_t frame_bytes = (size_t)B * SH * SW * 3, tensor_elems = (size_t)B * 3 * DH * DW;

    snprintf(path, sizeof path, "%s/frames.bin", dir);
    void* h_frames = slurp(path, frame_bytes);
    snprintf(path, sizeof path, "%s/logits1.bin", dir);
    void* h_l1 = slurp(path, sizeof(float) * R1 * C1);
    snprintf(path, sizeof path, "%s/logits2.bin", dir);
    void* h_l2 = slurp(path, sizeof(float) * R2 * C2);

    uint8_t* d_frames; float *d_tensor, *d_l1, *d_l2, *d_v1, *d_v2; int32_t *d_i1, *d_i2; void* d_ws = NULL;
    CHECK_CUDA(cudaMalloc((void**)&d_frames, frame_bytes));
    CHECK_CUDA(cudaMalloc((void**)&d_tensor, sizeof(float) * tensor_elems));
    CHECK_CUDA(cudaMalloc((void**)&d_l1, sizeof(float) * R1 * C1));
    CHECK_CUDA(cudaMalloc((void**)&d_l2, sizeof(float) * R2 * C2));
    CHECK_CUDA(cudaMalloc((void**)&d_v1, sizeof(float) * R1 * K1));
    CHECK_CUDA(cudaMalloc((void**)&d_i1, sizeof(int32_t) * R1 * K1));
    CHECK_CUDA(cudaMalloc((void**)&d_v2, sizeof(float) * R2 * K2));
    CHECK_CUDA(cudaMalloc((void**)&d_i2, sizeof(int32_t) * R2 * K2));
    CHECK_CUDA(cudaMemcpy(d_frames, h_frames, frame_bytes, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(d_l1, h_l1, sizeof(float) * R1 * C1, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(d_l2, h_l2, sizeof(float) * R2 * C2, cudaMemcpyHostToDevice));

    cudaStream_t stream;
    CHECK_CUDA(cudaStreamCreateWithFlags(&stream, cudaStreamNonBlocking));
    ws_preprocess_desc pre = {0};
    pre.src_w = SW; pre.src_h = SH; pre.src_row_stride = 3 * SW; pre.src_frame_stride = (int64_t)3 * SW * SH;
    pre.dst_w = DW; pre.dst_h = DH; pre.resize = WS_RESIZE_STRETCH; pre.pad_value = 114;
    pre.norm = WS_NORM_MEAN_STD;
    pre.mean[0] = 0.485f; pre.mean[1] = 0.456f; pre.mean[2] = 0.406f;
    pre.std[0] = 0.229f; pre.std[1] = 0.224f; pre.std[2] = 0.225f;
    pre.channel_order = WS_ORDER_RGB; pre.dst_type = WS_DTYPE_F32;
    CHECK_WS(ws_preprocess(&pre, d_frames, B, d_tensor, stream));

    size_t need1 = 0, need2 = 0;
    CHECK_WS(ws_topk_workspace_bytes(R1, C1, K1, &need1));
    CHECK_WS(ws_topk(d_l1, R1, C1, K1, d_v1, d_i1, NULL, 0, stream));
    CHECK_WS(ws_topk_workspace_bytes(R2, C2, K2, &need2));
    if (need1 != 0 || need2 == 0) { fprintf(stderr, "unexpected workspace sizes\n"); return 1; }
    CHECK_CUDA(cudaMalloc(&d_ws, need2));
    CHECK_WS(ws_topk_workspace_init(d_ws, need2, stream));
    for (int rep = 0; rep < 2; ++rep)   /* the workspace is ready again after each call */
        CHECK_WS(ws_topk(d_l2, R2, C2, K2, d_v2, d_i2, d_ws, need2, stream));
    CHECK_CUDA(cudaStreamSynchronize(stream));

    float* h_tensor = (float*)malloc(sizeof(float) * tensor_elems);
    float h_v1[R1 * K1], h_v2[R2 * K2];
    int32_t h_i1[R1 * K1], h_i2[R2 * K2];
    CHECK_CUDA(cudaMemcpy(h_tensor, d_tensor, sizeof(float) * tensor_elems, cudaMemcpyDeviceToHost));
    CHECK_CUDA(cudaMemcpy(h_v1, d_v1, sizeof h_v1, cudaMemcpyDeviceToHost));
    CHECK_CUDA(cudaMemcpy(h_i1, d_i1, sizeof h_i1, cudaMemcpyDeviceToHost));
    CHECK_CUDA(cudaMemcpy(h_v2, d_v2, sizeof h_v2, cudaMemcpyDeviceToHost));
    CHECK_CUDA(cudaMemcpy(h_i2, d_i2, sizeof h_i2, cudaMemcpyDeviceToHost));
    snprintf(path, sizeof path, "%s/tensor.bin", dir); dump(path, h_tensor, sizeof(float) * tensor_elems);
    snprintf(path, sizeof path, "%s/v1.bin", dir); dump(path, h_v1, sizeof h_v1);
    snprintf(path, sizeof path, "%s/i1.bin", dir); dump(path, h_i1, sizeof h_i1);
    snprintf(path, sizeof path, "%s/v2.bin", dir); dump(path, h_v2, sizeof h_v2);
    snprintf(path, sizeof path, "%s/i2.bin", dir); dump(path, h_i2, sizeof h_i2);
    printf("ok\n");
    return 0;
}
"""


def test_c_client_against_the_oracle(oracle, tmp_path):
    import __graft_entry__
    __graft_entry__.build()
    from post_processing_gb300 import binding
    lib_dir = os.path.dirname(binding.LIBRARY_PATH)
    cuda = "/usr/local/cuda"
    src = tmp_path / "client.c"
    src.write_text(CLIENT)
    exe = tmp_path / "client"
    subprocess.run(["gcc", "-std=c11", "-O1", "-I" + os.path.join(ROOT, "include"), "-I" + cuda + "/include",
                    str(src), "-o", str(exe), "-L" + lib_dir, "-l:libws.so", "-L" + cuda + "/lib64", "-lcudart",
                    "-Wl,-rpath," + lib_dir + ":" + cuda + "/lib64"], check=True)

    frames = synth.frames_uniform(4321, 3, 180, 320)
    l1 = synth.logits_with_ties(4322, 4, 1000)
    l2 = synth.logits_with_ties(4323, 2, 50000)
    frames.tofile(tmp_path / "frames.bin")
    l1.astype(np.float32).tofile(tmp_path / "logits1.bin")
    l2.astype(np.float32).tofile(tmp_path / "logits2.bin")
    run = subprocess.run([str(exe), str(tmp_path)], capture_output=True, text=True)
    assert run.returncode == 0, run.stderr
    assert run.stdout.strip() == "ok"

    tensor = np.fromfile(tmp_path / "tensor.bin", np.float32).reshape(3, 3, 96, 96)
    want = oracle.preprocess(frames, 320, 180, 96, 96)
    assert float(np.max(np.abs(tensor.astype(np.float64) - want))) <= 1e-5
    for (x, k, v, i) in ((l1, 5, "v1", "i1"), (l2, 32, "v2", "i2")):
        wv, wi = oracle.topk(x, k)
        gv = np.fromfile(tmp_path / f"{v}.bin", np.float32).reshape(x.shape[0], k)
        gi = np.fromfile(tmp_path / f"{i}.bin", np.int32).reshape(x.shape[0], k)
        assert np.array_equal(gi, wi)
        assert np.array_equal(gv.view(np.uint32), wv.view(np.uint32))
