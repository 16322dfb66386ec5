"""Pins of the oracle's step: reduction, AdamW, cast, sharding, buckets, skip.

See ``pins.py`` for what each check compares against.
"""
import pytest

import pins


@pytest.mark.parametrize("check", pins.ALL, ids=lambda f: f.__name__)
def test_pin(orc, check):
    check(orc)
