"""The C ABI without a GPU: libmsa.so builds for sm_103a, loads, exports
every function include/msa.h declares, sizes its workspaces, and rejects bad
arguments on the host before launching anything."""
import ctypes
import os
import re

import pytest

import block_sparse_attention_prefill_gb300 as msa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "msa.h")


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"MSA_API\s+[\w\s\*]*?\b(msa_\w+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    return msa.load()


def test_header_declares_the_calls():
    names = declared_functions()
    for n in ("msa_plan", "msa_prefill", "msa_decode", "msa_combine",
              "msa_plan_workspace_bytes", "msa_prefill_workspace_bytes",
              "msa_decode_workspace_bytes", "msa_read_status",
              "msa_status_string", "msa_version", "msa_read_counters"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    raw = ctypes.CDLL(msa.library_path())
    for n in declared_functions():
        assert hasattr(raw, n), n


def test_version_and_strings(lib):
    assert lib.msa_version() >= 100
    assert msa.status_string(0) == "ok"
    assert "workspace" in msa.status_string(4)


def test_workspace_sizes(lib):
    a = msa.plan_workspace_bytes(1, 2048, 16, 2, 8192, 2048)
    b = msa.plan_workspace_bytes(1, 4096, 16, 2, 8192, 4096)
    assert 0 < a < b
    # per (token, query head, slot): 128 E4M3 bytes of O and a 4-byte lse
    assert msa.prefill_workspace_bytes(2048, 16) >= 2048 * 16 * 16 * (128 + 4)
    assert msa.decode_workspace_bytes(64, 8, 16, 2, 131072) > 0


def _err(fn, *args):
    with pytest.raises(msa.MsaError) as e:
        fn(*args)
    return str(e.value)


def test_sizing_rejects_bad_shapes(lib):
    assert "unsupported" in _err(msa.plan_workspace_bytes, 1, 10, 6, 4, 8, 10)
    assert "unsupported" in _err(msa.plan_workspace_bytes, 1, 10, 256, 1, 8, 10)
    assert "out of range" in _err(msa.plan_workspace_bytes, -1, 10, 8, 1, 8, 10)
    assert "out of range" in _err(msa.decode_workspace_bytes, 4, 9, 16, 2, 1000)
    assert "out of range" in _err(msa.decode_workspace_bytes, 4, 8, 16, 2, 4)


def test_host_validation_before_launch(lib):
    P = ctypes.c_void_p
    plan = msa.MsaPlanStruct()
    fake = P(4096)  # never dereferenced: every call below fails on the host
    # NULL plan
    assert lib.msa_plan(fake, fake, fake, fake, 4, 8, 1, 10, 16, 2, 8, 10,
                        100, fake, 1 << 20, None, None) == 6
    # group size not an integer
    assert lib.msa_plan(fake, fake, fake, fake, 4, 8, 1, 10, 6, 4, 8, 10, 100,
                        fake, 1 << 20, ctypes.byref(plan), None) == 2
    # workspace too small
    assert lib.msa_plan(fake, fake, fake, fake, 4, 8, 1, 10, 16, 2, 8, 10, 100,
                        fake, 16, ctypes.byref(plan), None) == 4
    # max_seqlen_q above max_seqlen_k
    assert lib.msa_plan(fake, fake, fake, fake, 4, 8, 1, 10, 16, 2, 8, 200,
                        100, fake, 1 << 30, ctypes.byref(plan), None) == 1
    # block_table rows narrower than the pages of max_seqlen_k (300 keys: 3
    # pages, stride 2)
    assert lib.msa_plan(fake, fake, fake, fake, 2, 8, 1, 10, 16, 2, 8, 10, 300,
                        fake, 1 << 30, ctypes.byref(plan), None) == 1
    # misaligned workspace
    assert lib.msa_plan(fake, fake, fake, fake, 4, 8, 1, 10, 16, 2, 8, 10, 100,
                        P(4096 + 8), 1 << 30, ctypes.byref(plan), None) == 3
    # head shard: past the end of topk's heads, negative start; a range
    # that fits gets as far as the workspace check
    assert lib.msa_plan_heads(fake, 2, 1, fake, fake, fake, 4, 8, 1, 10, 16, 2, 8, 10,
                              100, fake, 1 << 30, ctypes.byref(plan), None) == 1
    assert lib.msa_plan_heads(fake, 2, -1, fake, fake, fake, 4, 8, 1, 10, 8, 1, 8, 10,
                              100, fake, 1 << 30, ctypes.byref(plan), None) == 1
    assert lib.msa_plan_heads(fake, 2, 1, fake, fake, fake, 4, 8, 1, 10, 8, 1, 8, 10,
                              100, fake, 16, ctypes.byref(plan), None) == 4
    # combine: bad split count, bad dtype
    assert lib.msa_combine(fake, 0, fake, 10, 0, fake, None, None) == 1
    assert lib.msa_combine(fake, 7, fake, 10, 4, fake, None, None) == 2
    assert lib.msa_combine(P(4100), 0, fake, 10, 4, fake, None, None) == 3
    # prefill: NULL plan
    assert lib.msa_prefill(fake, fake, 4, 1.0, 1.0, 1.0, 0.1, fake, 4, None,
                           fake, 1 << 20, fake, None, None) == 6
    # decode: n out of range
    assert lib.msa_decode(fake, fake, 4, 1.0, 1.0, 1.0, 0.1, fake, fake, 4,
                          fake, 2, 9, 16, 2, 1000, fake, 1 << 30, fake, None,
                          None, None) == 1
    # NVFP4 prefill: NULL plan; decode: n out of range
    assert lib.msa_prefill_nvfp4(fake, fake, 4, 1.0, 1.0, 1.0, 0.1, fake, 4,
                                 None, fake, 1 << 20, fake, None, None) == 6
    assert lib.msa_decode_nvfp4(fake, fake, 4, 1.0, 1.0, 1.0, 0.1, fake, fake,
                                4, fake, 2, 9, 16, 2, 1000, fake, 1 << 30,
                                fake, None, None, None) == 1
    # BF16-query prefill and its attention half: NULL plan
    assert lib.msa_prefill_bf16q(fake, fake, 4, 1.0, 1.0, 1.0, 0.1, fake, 4,
                                 None, fake, 1 << 20, fake, None, None) == 6
    assert lib.msa_prefill_attention_bf16q(fake, fake, 4, 1.0, 1.0, 1.0, 0.1, fake,
                                           4, None, fake, 1 << 20, None) == 6
    # NVFP4 -> E4M3 staging: negative count, NULL, misaligned; zero is a no-op
    assert lib.msa_nvfp4_to_e4m3(fake, -1, fake, None) == 1
    assert lib.msa_nvfp4_to_e4m3(None, 4, fake, None) == 6
    assert lib.msa_nvfp4_to_e4m3(P(4096 + 8), 4, fake, None) == 3
    assert lib.msa_nvfp4_to_e4m3(fake, 0, fake, None) == 0


def test_nvfp4_layout_constants():
    text = open(HEADER).read()
    slot = int(re.search(r"#define MSA_NVFP4_SLOT_BYTES (\d+)", text).group(1))
    ph = int(re.search(r"#define MSA_NVFP4_PAGE_HEAD_BYTES (\d+)", text).group(1))
    # 128 tokens x (64 code bytes + 8 block scales); K slot + V slot
    assert slot == 128 * 64 + 128 * 8 == msa.NVFP4_SLOT_BYTES
    assert ph == 2 * slot


def test_binding_rejects_host_tensors_and_wrong_pools():
    # argument checks in the Python binding run before any library call
    import torch
    kv4 = torch.zeros((2, 1, 2, msa.NVFP4_SLOT_BYTES), dtype=torch.uint8)
    assert "CUDA" in _err(msa.msa_nvfp4_to_e4m3, kv4)
    assert "dtype" in _err(msa._need, kv4.to(torch.int16), "kv4", (torch.uint8,),
                           False)


def test_decode_bindings_check_shapes_before_the_library():
    # the library sees only pointers: a pool for the wrong number of KV heads
    # or an undersized output would be read or written out of bounds on the
    # device, so the bindings refuse them first (host tensors suffice here:
    # the shape checks come before the device checks)
    import torch
    B, n, Hq, Hkv = 3, 4, 16, 2
    q = torch.zeros((B * n, Hq, 128), dtype=torch.uint8)
    topk = torch.zeros((B * n, Hkv, 16), dtype=torch.int32)
    bt = torch.zeros((B, 8), dtype=torch.int32)
    seq = torch.full((B,), 900, dtype=torch.int32)
    kv_bad = torch.zeros((8, Hkv + 1, 128, 256), dtype=torch.uint8)
    out = torch.zeros((B * n, Hq, 128), dtype=torch.bfloat16)
    out_small = torch.zeros((B * n - 1, Hq, 128), dtype=torch.bfloat16)
    lse_bad = torch.zeros((B * n, Hq + 1), dtype=torch.float32)
    kv = torch.zeros((8, Hkv, 128, 256), dtype=torch.uint8)
    args = (1.0, 1.0, 1.0, 0.1)
    assert "kv must be" in _err(msa.msa_decode_noalloc, q, kv_bad, *args, topk,
                                bt, seq, n, 1000, out, None)
    assert "out must be" in _err(msa.msa_decode_noalloc, q, kv, *args, topk,
                                 bt, seq, n, 1000, out_small, None)
    assert "lse must be" in _err(msa.msa_decode_noalloc, q, kv, *args, topk,
                                 bt, seq, n, 1000, out, lse_bad)
    assert "B*n rows" in _err(msa.msa_decode_noalloc, q[:-1], kv, *args, topk,
                              bt, seq, n, 1000, out, None)
    assert "out is required" in _err(msa.msa_decode_noalloc, q, kv, *args,
                                     topk, bt, seq, n, 1000, None, None)
    assert "kv must be" in _err(msa.msa_decode, q, kv_bad, *args, topk, bt,
                                seq, n, 1000)
    assert "out must be" in _err(msa.msa_decode, q, kv, *args, topk, bt, seq,
                                 n, 1000, None, out_small)
