"""The C-ABI library without a GPU: it loads, exports every function that
include/qp.h declares, and rejects bad arguments on the host before anything
is launched (no compute call is made here)."""
import ctypes
import os
import re
import subprocess

import pytest

import block_quantized_weight_qp_gb300 as qp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "qp.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(qp_\w+)\s*\(", text)))


def test_header_declares_the_binding_exports():
    assert declared_functions() == sorted(qp.EXPORTS)


def test_library_exports_every_declared_symbol():
    lib = qp.load()
    for name in declared_functions():
        assert hasattr(lib, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", qp.library_path()], capture_output=True, text=True).stdout
    exported = set(line.split()[-1] for line in out.splitlines() if line.strip())
    for name in declared_functions():
        assert name in exported, name


def test_library_is_built_for_sm_103a_only():
    out = subprocess.run(["cuobjdump", "--list-elf", qp.library_path()], capture_output=True, text=True).stdout
    arches = set(re.findall(r"sm_\d+a?", out))
    assert arches == {"sm_103a"}, arches


def test_block_info_and_row_bytes():
    assert qp.qp_block_info(qp.Q8_0) == (32, 34)
    assert qp.qp_block_info(qp.Q4_K) == (256, 144)
    assert qp.qp_block_info(qp.Q2_K) == (256, 84)
    assert qp.qp_block_info(qp.Q6_K) == (256, 210)
    assert qp.qp_row_bytes(qp.Q4_K, 1000) == 4 * 144
    assert qp.qp_row_bytes(qp.Q8_0, 33) == 2 * 34
    assert qp.qp_block_info(qp.Q5_K) == (256, 176) and qp.qp_block_info(qp.F16) == (1, 2)
    assert qp.qp_row_bytes(qp.F16, 1000) == 2000 and qp.qp_row_bytes(qp.Q5_K, 300) == 2 * 176
    assert qp.qp_row_bytes(11, 256) == -1 and qp.qp_row_bytes(qp.Q4_K, 0) == -1
    with pytest.raises(qp.QPError) as e:
        qp.qp_block_info(21)
    assert e.value.status == qp.QP_ERR_UNSUPPORTED_TYPE


def test_status_strings():
    lib = qp.load()
    names = set()
    for s in range(9):
        assert lib.qp_status_str(s)
        names.add(lib.qp_status_str(s))
    assert len(names) == 9                       # every status has its own description
    assert lib.qp_status_str(9) == b"unknown status"
    assert qp.status_str(qp.QP_ERR_TIMEOUT) == "device-side wait timed out"
    assert "tensor-memory" in qp.status_str(qp.QP_ERR_PAIR_ALLOC)


FAKE = 1 << 40  # 16-byte aligned, never dereferenced: every call below fails its host check


@pytest.mark.parametrize("call,status", [
    (lambda l: l.qp_dequant_f32(qp.Q4_K, None, 4, 256, FAKE, None), qp.QP_ERR_INVALID_PARAMETER),
    (lambda l: l.qp_dequant_f32(qp.Q4_K, FAKE, 0, 256, FAKE, None), qp.QP_ERR_INVALID_PARAMETER),
    (lambda l: l.qp_dequant_f16(qp.Q4_K, FAKE, 4, -1, FAKE, None), qp.QP_ERR_INVALID_PARAMETER),
    (lambda l: l.qp_dequant_f32(11, FAKE, 4, 256, FAKE, None), qp.QP_ERR_UNSUPPORTED_TYPE),
    (lambda l: l.qp_dequant_f16(qp.Q6_K, FAKE + 2, 4, 256, FAKE, None), qp.QP_ERR_MISALIGNED),
    (lambda l: l.qp_prefill_gemm(qp.Q4_K, FAKE, 256, 256, FAKE, 0, FAKE, None), qp.QP_ERR_INVALID_PARAMETER),
    (lambda l: l.qp_prefill_gemm(qp.Q4_K, FAKE, 256, 1000, FAKE, 16, FAKE, None), qp.QP_ERR_UNSUPPORTED_SHAPE),
    (lambda l: l.qp_prefill_gemm(qp.Q4_K, FAKE, 258, 256, FAKE, 16, FAKE, None), qp.QP_ERR_UNSUPPORTED_SHAPE),
    (lambda l: l.qp_prefill_gemm(qp.Q2_K, FAKE, 256, 512, FAKE, 16, FAKE, None), qp.QP_ERR_UNSUPPORTED_SHAPE),
    (lambda l: l.qp_prefill_gemm(qp.Q6_K, FAKE, 256, 1024, FAKE, 16, FAKE, None), qp.QP_ERR_UNSUPPORTED_SHAPE),
    (lambda l: l.qp_prefill_gemm(3, FAKE, 256, 256, FAKE, 16, FAKE, None), qp.QP_ERR_UNSUPPORTED_TYPE),
    (lambda l: l.qp_prefill_gemm(qp.Q4_K, FAKE, 256, 256, FAKE + 8, 16, FAKE, None), qp.QP_ERR_MISALIGNED),
    (lambda l: l.qp_prefill_gemm_f16w(None, 256, 256, FAKE, 16, FAKE, None), qp.QP_ERR_INVALID_PARAMETER),
    (lambda l: l.qp_prefill_gemm_f16w(FAKE, 256, 100, FAKE, 16, FAKE, None), qp.QP_ERR_UNSUPPORTED_SHAPE),
    (lambda l: l.qp_prefill_chunked(qp.Q4_K, FAKE, None, 256, 256, FAKE, 16, FAKE, 0, 0, None),
     qp.QP_ERR_INVALID_PARAMETER),
    (lambda l: l.qp_prefill_chunked(qp.Q4_K, FAKE, None, 256, 256, FAKE, 16, FAKE, 8, 2, None),
     qp.QP_ERR_INVALID_PARAMETER),
    (lambda l: l.qp_prefill_chunked(qp.Q4_K, FAKE, None, 256, 256, FAKE, 16, FAKE, 8, 1, None),
     qp.QP_ERR_INVALID_PARAMETER),
])
def test_host_side_argument_checks(call, status):
    assert call(qp.load()) == status


def descs(*shapes, W=FAKE, X=FAKE, Y=FAKE):
    arr = (qp.QPGemmDesc * max(len(shapes), 1))()
    for k, (out_f, in_f) in enumerate(shapes):
        arr[k] = qp.QPGemmDesc(W, out_f, in_f, X, Y)
    return arr


@pytest.mark.parametrize("call,status", [
    (lambda l: l.qp_prefill_gemm_group(qp.Q4_K, None, 1, 16, None), qp.QP_ERR_INVALID_PARAMETER),
    (lambda l: l.qp_prefill_gemm_group(qp.Q4_K, descs((256, 256)), 0, 16, None), qp.QP_ERR_INVALID_PARAMETER),
    (lambda l: l.qp_prefill_gemm_group(qp.Q4_K, descs(*[(256, 256)] * 9), 9, 16, None),
     qp.QP_ERR_INVALID_PARAMETER),
    (lambda l: l.qp_prefill_gemm_group(3, descs((256, 256)), 1, 16, None), qp.QP_ERR_UNSUPPORTED_TYPE),
    (lambda l: l.qp_prefill_gemm_group(qp.Q4_K, descs((256, 256)), 1, 0, None), qp.QP_ERR_INVALID_PARAMETER),
    (lambda l: l.qp_prefill_gemm_group(qp.Q4_K, descs((256, 256), (256, 1000)), 2, 16, None),
     qp.QP_ERR_UNSUPPORTED_SHAPE),
    (lambda l: l.qp_prefill_gemm_group(qp.Q2_K, descs((256, 1024), (256, 512)), 2, 16, None),
     qp.QP_ERR_UNSUPPORTED_SHAPE),
    (lambda l: l.qp_prefill_gemm_group(0, descs((256, 256), (256, 100)), 2, 16, None),
     qp.QP_ERR_UNSUPPORTED_SHAPE),
    (lambda l: l.qp_prefill_gemm_group(qp.Q8_0, descs((256, 256), W=None), 1, 16, None),
     qp.QP_ERR_INVALID_PARAMETER),
    (lambda l: l.qp_prefill_gemm_group(qp.Q8_0, descs((256, 256), (128, 256), Y=FAKE + 4), 2, 16, None),
     qp.QP_ERR_MISALIGNED),
    (lambda l: l.qp_prefill_chunked_group(qp.Q4_K, descs((256, 256)), 1, 16, 0, None), qp.QP_ERR_INVALID_PARAMETER),
    (lambda l: l.qp_prefill_chunked_group(qp.Q4_K, descs((256, 256)), 0, 16, 8, None), qp.QP_ERR_INVALID_PARAMETER),
    (lambda l: l.qp_prefill_chunked_group(0, descs((256, 300)), 1, 16, 8, None), qp.QP_ERR_UNSUPPORTED_SHAPE),
])
def test_grouped_call_argument_checks(call, status):
    assert call(qp.load()) == status


@pytest.mark.parametrize("call,status", [
    (lambda l: l.qp_decode_gemv(qp.Q4_K, None, 256, 256, FAKE, 1, FAKE, None), qp.QP_ERR_INVALID_PARAMETER),
    (lambda l: l.qp_decode_gemv(qp.Q4_K, FAKE, 256, 256, FAKE, 0, FAKE, None), qp.QP_ERR_INVALID_PARAMETER),
    (lambda l: l.qp_decode_gemv(qp.Q4_K, FAKE, 0, 256, FAKE, 1, FAKE, None), qp.QP_ERR_INVALID_PARAMETER),
    (lambda l: l.qp_decode_gemv(11, FAKE, 256, 256, FAKE, 1, FAKE, None), qp.QP_ERR_UNSUPPORTED_TYPE),
    (lambda l: l.qp_decode_gemv(qp.Q4_K, FAKE, 256, 256, FAKE, 9, FAKE, None), qp.QP_ERR_UNSUPPORTED_SHAPE),
    (lambda l: l.qp_decode_gemv(qp.Q4_K, FAKE, 256, 288, FAKE, 1, FAKE, None), qp.QP_ERR_UNSUPPORTED_SHAPE),
    (lambda l: l.qp_decode_gemv(qp.Q8_0, FAKE, 256, 48, FAKE, 1, FAKE, None), qp.QP_ERR_UNSUPPORTED_SHAPE),
    (lambda l: l.qp_decode_gemv(qp.F16, FAKE, 256, (1 << 24) + 32, FAKE, 8, FAKE, None), qp.QP_ERR_UNSUPPORTED_SHAPE),
    (lambda l: l.qp_decode_gemv(qp.Q8_0, FAKE + 8, 256, 64, FAKE, 1, FAKE, None), qp.QP_ERR_MISALIGNED),
    (lambda l: l.qp_decode_gemv(qp.Q8_0, FAKE, 256, 64, FAKE, 1, FAKE + 2, None), qp.QP_ERR_MISALIGNED),
    (lambda l: l.qp_decode_gemv_group(qp.Q4_K, None, 1, 1, None), qp.QP_ERR_INVALID_PARAMETER),
    (lambda l: l.qp_decode_gemv_group(qp.Q4_K, descs((256, 256)), 0, 1, None), qp.QP_ERR_INVALID_PARAMETER),
    (lambda l: l.qp_decode_gemv_group(qp.Q4_K, descs(*[(256, 256)] * 9), 9, 1, None), qp.QP_ERR_INVALID_PARAMETER),
    (lambda l: l.qp_decode_gemv_group(qp.Q4_K, descs((256, 256), (256, 288)), 2, 1, None),
     qp.QP_ERR_UNSUPPORTED_SHAPE),
    (lambda l: l.qp_decode_gemv_group(qp.Q4_K, descs((256, 256)), 1, 9, None), qp.QP_ERR_UNSUPPORTED_SHAPE),
    (lambda l: l.qp_decode_gemv_group(11, descs((256, 256)), 1, 1, None), qp.QP_ERR_UNSUPPORTED_TYPE),
])
def test_decode_gemv_argument_checks(call, status):
    assert call(qp.load()) == status


def test_no_device_is_an_error_not_a_fallback():
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    lib = qp.load()
    assert lib.qp_dequant_f32(qp.Q4_K, FAKE, 4, 256, FAKE, None) == qp.QP_ERR_NO_DEVICE
    assert lib.qp_prefill_gemm(qp.Q4_K, FAKE, 256, 256, FAKE, 16, FAKE, None) == qp.QP_ERR_NO_DEVICE
    assert lib.qp_prefill_gemm_group(qp.Q4_K, descs((256, 256), (512, 512)), 2, 16, None) == qp.QP_ERR_NO_DEVICE
    assert lib.qp_decode_gemv(qp.Q4_K, FAKE, 256, 256, FAKE, 1, FAKE, None) == qp.QP_ERR_NO_DEVICE
    assert lib.qp_decode_gemv_group(qp.Q4_K, descs((256, 256), (64, 512)), 2, 1, None) == qp.QP_ERR_NO_DEVICE
