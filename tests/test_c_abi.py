"""The boundary is a plain C ABI: a C program built against include/sa_api.h and linked to
libsa.so calls the host-only entry points and the argument checks (no GPU needed)."""
import os
import shutil
import subprocess

import pytest

import content_adaptive_sparse_gb300 as sa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_c_client_links_and_runs(tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    lib = sa.build_library()
    exe = tmp_path / "abi_smoke"
    subprocess.run([cc, "-std=c99", "-O1", "-I", os.path.join(ROOT, "include"),
                    os.path.join(ROOT, "tests", "c", "abi_smoke.c"), "-o", str(exe),
                    "-L", os.path.dirname(lib), "-lsa", "-Wl,-rpath," + os.path.dirname(lib)],
                   check=True, capture_output=True, text=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert out.returncode == 0, out.stderr
    assert "c abi ok" in out.stdout


@pytest.mark.gpu
def test_c_client_runs_the_hot_path_on_the_gpu(tmp_path):
    """A C program (tests/c/abi_gpu.c) runs sa_build_mask and sa_attn_fwd on the tiny
    compression-guided workload through the C header alone; its CSR must equal the
    oracle's bit for bit and its O / LSE must be within the attention tolerance."""
    import numpy as np

    import oracle
    from oracle import masks as om
    from workloads import bf16_bits_to_f64, byte_stream, qkv_bits, workload
    from gpu_helpers import assert_attention_close, torch_cuda

    torch_cuda()
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    lib = sa.build_library()
    cuda_home = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    exe = tmp_path / "abi_gpu"
    subprocess.run([cc, "-std=c99", "-O1", "-I", os.path.join(ROOT, "include"), "-I",
                    os.path.join(cuda_home, "include"), os.path.join(ROOT, "tests", "c", "abi_gpu.c"), "-o", str(exe),
                    "-L", os.path.dirname(lib), "-lsa", "-L", os.path.join(cuda_home, "lib64"), "-lcudart",
                    "-lm", "-Wl,-rpath," + os.path.dirname(lib), "-Wl,-rpath," + os.path.join(cuda_home, "lib64")],
                   check=True, capture_output=True, text=True)
    cfg = workload("tiny_topk")
    data = byte_stream(cfg)
    ratios = oracle.block_ratios(data, cfg["block"]).astype(np.float32)
    qb, kb, vb = qkv_bits(cfg, q_scale_pow2=2)
    bt, n, h, hkv, d, b = (cfg[k] for k in ("batch", "n_tokens", "heads", "kv_heads", "head_dim", "block"))
    hdr = np.array([bt, n, h, hkv, d, b, cfg["window_blocks"], cfg["global_blocks"], cfg["topk"]], dtype=np.int32)
    prob = tmp_path / "problem.bin"
    with open(prob, "wb") as fh:
        for arr in (hdr, ratios, qb, kb, vb):
            fh.write(np.ascontiguousarray(arr).tobytes())
    res = tmp_path / "result.bin"
    out = subprocess.run([str(exe), str(prob), str(res)], capture_output=True, text=True, timeout=120)
    assert out.returncode == 0, out.stderr
    raw = res.read_bytes()
    nb = n // b
    pos = 0
    rp = np.frombuffer(raw, dtype=np.int32, count=bt * (nb + 1), offset=pos).reshape(bt, nb + 1)
    pos += rp.nbytes
    nnz = int(np.frombuffer(raw, dtype=np.int32, count=1, offset=pos)[0])
    pos += 4
    ci = np.frombuffer(raw, dtype=np.int32, count=nnz, offset=pos)
    pos += ci.nbytes
    o_bits = np.frombuffer(raw, dtype=np.uint16, count=bt * n * h * d, offset=pos).reshape(bt, n, h, d)
    pos += o_bits.nbytes
    lse = np.frombuffer(raw, dtype=np.float32, count=bt * h * n, offset=pos).reshape(bt, h, n)
    p = om.MaskParams("topk", b, n, 1, cfg["window_blocks"], cfg["global_blocks"], cfg["topk"])
    rp_o, ci_o = om.build_csr(p, ratios, bt)
    assert np.array_equal(rp, rp_o) and np.array_equal(ci, ci_o)
    o_ref, lse_ref = oracle.attention_csr(bf16_bits_to_f64(qb), bf16_bits_to_f64(kb), bf16_bits_to_f64(vb), rp_o,
                                          ci_o, b, 1)
    assert_attention_close(bf16_bits_to_f64(o_bits), lse.astype(np.float64), o_ref, lse_ref, "C client")
