"""CPU oracle of the dense prefill indexer -- test infrastructure only.

Imported by the tests, the smoke check and the benchmark's CPU baseline;
never by the product package.
"""
