"""CPU oracle package: test infrastructure only (tests, smoke check, bench CPU baseline)."""
