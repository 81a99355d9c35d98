"""The C ABI used from plain C: tests/c_abi_client.c includes include/h3attn.h, links
libh3attn.so and the CUDA runtime, and runs tagged RoPE (with a continuation start frame) and
packed varlen attention with no Python in between.

* CPU: the header compiles as strict C11 and the client links against the library.
* GPU: the client's outputs are the very bytes the Python binding produces for the same inputs
  (the binding only marshals arguments), pad rows stay untouched, and the result agrees with the
  oracle's fp64 RoPE + attention from the raw Q/K.
"""
import glob
import os
import shutil
import subprocess

import numpy as np
import pytest
import torch

import oracle
import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CLIENT_SRC = os.path.join(ROOT, "tests", "c_abi_client.c")


def _cuda_root():
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return os.path.dirname(os.path.dirname(os.path.realpath(cand)))
    pytest.skip("no CUDA toolkit")


def _compile_client(out_dir):
    import __graft_entry__

    __graft_entry__.build()
    import packed_varlen_attention_modality_gb300 as h3

    cuda = _cuda_root()
    libdirs = [d for d in [os.path.join(cuda, "lib64")] + glob.glob(os.path.join(cuda, "targets", "*", "lib"))
               if os.path.exists(os.path.join(d, "libcudart.so"))]
    assert libdirs, "libcudart.so not found under " + cuda
    pkg = os.path.dirname(h3.lib_path())
    exe = os.path.join(str(out_dir), "c_abi_client")
    cmd = ["gcc", "-std=c11", "-O2", "-Wall", "-Wextra", "-pedantic", CLIENT_SRC,
           "-I" + os.path.join(ROOT, "include"), "-I" + os.path.join(cuda, "include"),
           "-L" + pkg, "-l:" + os.path.basename(h3.lib_path()), "-L" + libdirs[0], "-lcudart",
           "-Wl,-rpath," + pkg + ":" + libdirs[0], "-o", exe]
    r = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    assert r.returncode == 0, " ".join(cmd) + "\n" + r.stdout
    return exe, r.stdout


def test_header_compiles_as_c11_and_client_links(tmp_path):
    exe, log = _compile_client(tmp_path)
    assert os.path.exists(exe)
    assert "h3attn.h" not in log, log  # no diagnostics from the public header


def _write_input(path, wl):
    C, H, D = wl.q.shape
    N, S, R = wl.num_tokens, wl.num_segments, len(wl.start_frames)
    with open(path, "wb") as f:
        np.asarray([C, H, D, N, S, R, max(1, int(np.diff(wl.cu_seqlens).max()))], np.int32).tofile(f)
        for t in (wl.q, wl.k, wl.v):
            t.contiguous().view(torch.int16).numpy().tofile(f)
        np.asarray(wl.pos[:N], np.float32).tofile(f)
        np.asarray(wl.tag[:N], np.uint8).tofile(f)
        np.asarray(wl.cu_seqlens, np.int32).tofile(f)
        np.asarray(wl.cu_requests, np.int32).tofile(f)
        np.asarray(wl.start_frames, np.float32).tofile(f)


def _read_output(path, wl):
    C, H, D = wl.q.shape
    raw = np.fromfile(path, dtype=np.uint8)
    st = raw[:12].view(np.int32)
    o_bytes = C * H * D * 2
    o = torch.from_numpy(raw[12:12 + o_bytes].copy().view(np.int16)).view(torch.bfloat16).view(C, H, D)
    lse = torch.from_numpy(raw[12 + o_bytes:].copy().view(np.float32)).view(H, C)
    return st, o, lse


@pytest.mark.gpu
@pytest.mark.parametrize("case", ["worked_example", "single_request_4096"])
def test_c_client_equals_binding_and_oracle(tmp_path, case):
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    if case == "worked_example":
        wl = W.tiny_example(capacity=64)
        wl.start_frames = np.asarray([238.0], np.float32)  # the pages' printed start frame
    else:
        wl = W.single_request_4k(capacity=4160)
        wl.start_frames = np.asarray([119.0], np.float32)
    exe, _ = _compile_client(tmp_path)
    inp, outp = os.path.join(str(tmp_path), "in.bin"), os.path.join(str(tmp_path), "out.bin")
    _write_input(inp, wl)
    r = subprocess.run([exe, inp, outp], stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True,
                       timeout=300)
    assert r.returncode == 0, r.stdout
    st, o_c, lse_c = _read_output(outp, wl)
    assert st.tolist() == [0, 0, 0], r.stdout

    # the same calls through the Python binding
    import packed_varlen_attention_modality_gb300 as h3

    dev = torch.device("cuda", 0)
    N, (C, H, D) = wl.num_tokens, wl.q.shape
    q, k, v = (t.to(dev) for t in (wl.q, wl.k, wl.v))
    pos, tag = torch.from_numpy(wl.pos[:N]).to(dev), torch.from_numpy(wl.tag[:N]).to(dev)
    cu, cu_req = torch.from_numpy(wl.cu_seqlens).to(dev), torch.from_numpy(wl.cu_requests).to(dev)
    frames = torch.from_numpy(wl.start_frames).to(dev)
    qr, kr = q.clone(), k.clone()
    h3.rope_apply(q, k, pos, tag, cu_req, frames, num_tokens=N, q_out=qr, k_out=kr)
    o = torch.full_like(q, 3.0)
    lse = torch.full((H, C), 5.0, device=dev)
    maxs = max(1, int(np.diff(wl.cu_seqlens).max()))
    ws = torch.empty(max(16, h3.varlen_attn_workspace_size(wl.num_segments, H, maxs, D)), dtype=torch.uint8,
                     device=dev)
    h3.varlen_attn_fwd(qr, kr, v, cu, maxs, out=o, lse=lse, workspace=ws)
    torch.cuda.synchronize()
    assert h3.get_device_error(dev) == 0
    assert torch.equal(o.cpu(), o_c) and torch.equal(lse.cpu(), lse_c), "C client and binding differ"
    assert torch.all(o_c[N:] == 3.0) and torch.all(lse_c[:, N:] == 5.0)

    # and the oracle from the raw Q/K (its own fp64 RoPE with the time shift), every row
    qo = oracle.rope_apply(wl.q, wl.pos, wl.tag, wl.cu_requests, wl.start_frames, num_tokens=N)
    ko = oracle.rope_apply(wl.k, wl.pos, wl.tag, wl.cu_requests, wl.start_frames, num_tokens=N)
    ref_o, _ = oracle.varlen_attention(qo[:N], ko[:N], wl.v[:N].double().numpy(), wl.cu_seqlens)
    err = np.abs(o_c[:N].float().numpy().astype(np.float64) - ref_o[:N])
    assert err.max() <= 2e-2 and err.mean() <= 2e-3, f"{case}: max {err.max():.3e} mean {err.mean():.3e}"
