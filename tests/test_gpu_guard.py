"""The guard-band harness itself (tests/guard.py): a write just past the end
of a banded buffer, made here with an ordinary in-bounds torch write into the
band, is reported by the check that runs after every GPU test."""
import pytest
import torch

import guard

pytestmark = pytest.mark.gpu


def test_a_write_into_a_band_is_reported():
    t = guard.guarded(torch.arange(100, dtype=torch.int32, device="cuda"), "probe")
    guard.check_and_release()  # intact
    raw = torch.empty(0, dtype=torch.uint8, device="cuda").set_(t.untyped_storage())
    n = t.numel() * t.element_size()
    for pos in (guard.GUARD + n, guard.GUARD - 1):  # first byte after, last byte before
        saved = int(raw[pos].item())
        raw[pos] = 0
        with pytest.raises(AssertionError, match="probe"):
            guard.check_and_release()
        raw[pos] = saved
    guard.check_and_release()
    assert torch.equal(t, torch.arange(100, dtype=torch.int32, device="cuda"))
