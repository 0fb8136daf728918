"""The failure path of the library's bounded device waits, exercised without any fault: a kernel
whose mbarrier wait cannot complete gives up after its limit, records the event in the device error
word and ends normally; the host reads KVARN_ERR_TIMEOUT and the device keeps working."""
import time

import pytest
import torch

pytestmark = pytest.mark.gpu


def test_wait_that_runs_out_is_reported_and_the_device_stays_usable(kv):
    torch.cuda.synchronize()
    assert kv.kvarn_device_error() == 0  # start from clear error words
    t0 = time.perf_counter()
    kv.kvarn_check_bounded_wait(1000)  # 1 ms limit
    with pytest.raises(kv.KvarnError) as ei:
        kv.kvarn_device_error()  # synchronises: the kernel has returned by now
    elapsed = time.perf_counter() - t0
    assert ei.value.status == kv.KVARN_ERR_TIMEOUT
    assert ei.value.code == 8  # bit 4: the self-check's wait, nothing else
    assert elapsed < 5.0, f"the 1 ms wait took {elapsed:.2f} s to give up"
    # read and cleared: a second read is clean
    assert kv.kvarn_device_error() == 0
    # the context is intact: an encode right after runs and reports no error
    cfg = kv.kvarn_config_from_preset("kvarn_k2v2_g128")
    x = kv.synthetic.outlier_kv(3, 2, 128, device="cuda")[0].reshape(2, 128, 128)
    codes = torch.empty(2, 4096, dtype=torch.uint8, device="cuda")
    params = torch.empty(2, 512, dtype=torch.uint8, device="cuda")
    scale = torch.zeros(2, device="cuda")
    kv.kvarn_encode_blocks(cfg, kv.KVARN_KIND_K, x, codes, params, scale)
    torch.cuda.synchronize()
    assert kv.kvarn_device_error() == 0
    assert torch.all(scale > 0)


def test_two_checks_in_a_row_each_report_once(kv):
    assert kv.kvarn_device_error() == 0
    for _ in range(2):
        kv.kvarn_check_bounded_wait(200)
        with pytest.raises(kv.KvarnError) as ei:
            kv.kvarn_device_error()
        assert ei.value.code == 8
    assert kv.kvarn_device_error() == 0
