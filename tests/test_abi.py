"""The C-ABI library loads on a machine without a GPU and exports every entry
point that include/nc.h declares; host-only checks need no device."""
import ctypes
import os
import re

import pytest

from transformer_forward_gpt_b300 import binding, build, synth

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "nc.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.load()


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"NC_API\s+[\w\s\*]+?\b(nc_\w+)\s*\(", text)))


def test_header_declares_entry_points():
    names = declared_symbols()
    for want in ("nc_model_create", "nc_prefill", "nc_decode_step", "nc_kv_cache_alloc"):
        assert want in names
    assert set(names) == set(binding.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_only_nc_symbols_are_exported(lib):
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", binding.LIB_PATH], capture_output=True,
                         text=True).stdout
    names = [l.split()[-1] for l in out.splitlines() if " T " in l]
    assert names and all(n.startswith("nc_") for n in names), names


def test_param_count_matches_microgpt_shape(lib):
    cfg = binding.make_config(synth.TINY, 16, 1)
    assert binding.nc_param_count(cfg) == synth.param_count(synth.TINY) == 3936
    for s in (synth.D12, synth.D20, synth.D20_MQA, synth.D26):
        assert binding.nc_param_count(binding.make_config(s, 16, 1)) == synth.param_count(s)


def test_kv_cache_bytes(lib):
    cfg = binding.make_config(synth.D20_MQA, 1152, 32)
    per = 20 * 32 * 1 * 1152 * 128 * 2
    assert binding.nc_kv_cache_bytes(cfg, 32, 1152) == 256 + 2 * per


def test_create_rejects_bad_config_without_touching_the_device(lib):
    bad = binding.make_config(synth.with_changes(synth.D20, n_kv_head=3), 16, 1)
    with pytest.raises(binding.NcError) as e:
        binding.nc_model_create(bad, 0, 0, [(0,) * 6] * bad.n_layer)
    assert e.value.code == binding.NC_ERR_INVALID_ARG
    bad = binding.make_config(synth.with_changes(synth.D20, head_dim=64), 16, 1)
    with pytest.raises(binding.NcError) as e:
        binding.nc_model_create(bad, 0, 0, [(0,) * 6] * bad.n_layer)
    assert e.value.code == binding.NC_ERR_UNSUPPORTED
    assert "head_dim" in binding.load().nc_last_error().decode()


def test_status_strings(lib):
    assert lib.nc_status_string(0) == b"ok"
    assert lib.nc_status_string(binding.NC_ERR_BOUNDS) == b"token id out of range"
    assert lib.nc_status_string(binding.NC_ERR_RANGE) == b"value out of fp16 range"
    assert binding.nc_version().startswith("nc-b300")


def test_sample_and_continue_reject_bad_arguments_on_the_host(lib):
    """Argument checks of nc_op_sample and nc_prefill_continue happen before any
    device call (no GPU needed); zero rows is a valid empty call."""
    fake = 1 << 20   # never dereferenced: the checks return first
    for args in [(None, 2, 8, 1.0, fake, fake), (fake, 2, 8, 1.0, None, fake),
                 (fake, 2, 8, 1.0, fake, None), (fake, 2, 0, 1.0, fake, fake),
                 (fake, -1, 8, 1.0, fake, fake)]:
        with pytest.raises(binding.NcError) as e:
            binding.nc_op_sample(*args, stream=0)
        assert e.value.code == binding.NC_ERR_INVALID_ARG
    binding.nc_op_sample(fake, 0, 8, 0.7, fake, fake, stream=0)   # no rows: nothing to do
    with pytest.raises(binding.NcError) as e:
        binding.nc_prefill_continue(None, fake, 1, 4, fake, None, stream=0)
    assert e.value.code == binding.NC_ERR_INVALID_ARG


def test_cross_entropy_scratch_and_host_checks(lib):
    """Scratch of nc_op_cross_entropy: the per-block pairs (8 bytes per row and
    256-column block) and two per-row arrays, each rounded up to 256 bytes; the
    argument checks of the loss entry points return before any device call."""
    def r256(x):
        return (x + 255) // 256 * 256
    for M, N in [(1, 1), (300, 1000), (8192, 65536), (37, 257)]:
        want = r256(M * ((N + 255) // 256) * 8) + 2 * r256(M * 4)
        assert binding.nc_op_cross_entropy_scratch_bytes(M, N) == want
    assert binding.nc_op_cross_entropy_scratch_bytes(4, 0) == 0
    assert binding.nc_op_cross_entropy_scratch_bytes(-1, 8) == 0
    fake = 1 << 20   # 16-byte aligned, never dereferenced: the checks return first
    ok = (fake, fake, fake, 4, 256, 64, binding.NC_BF16, None, fake, fake, 1 << 20)
    for i, bad in [(2, None), (2, fake + 2), (8, None), (3, -1), (5, 0),
                   (6, binding.NC_F32), (10, 16)]:
        args = list(ok)
        args[i] = bad
        with pytest.raises(binding.NcError) as e:
            binding.nc_op_cross_entropy(*args, stream=0)
        assert e.value.code == binding.NC_ERR_INVALID_ARG, (i, bad)
    args = list(ok)
    args[5] = 48                                   # K not a multiple of 64
    with pytest.raises(binding.NcError) as e:
        binding.nc_op_cross_entropy(*args, stream=0)
    assert e.value.code == binding.NC_ERR_UNSUPPORTED
    with pytest.raises(binding.NcError) as e:
        binding.nc_prefill_loss(None, fake, fake, 1, 4, None, fake, None, stream=0)
    assert e.value.code == binding.NC_ERR_INVALID_ARG
